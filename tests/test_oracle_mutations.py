"""The oracle pins must fail when a plausible mistake is planted in the oracle.

Each case copies the oracle into a temporary tree, applies one textual
mutation on the CPU (a dropped smoothing term, a wrong normaliser, a flipped
sign, a missing max-subtraction, a missing mask) and runs the pin suite
against the mutated copy; at least one pin has to fail.
"""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTATIONS = [
    ("drop smoothing row-sum term",
     "loss = loss - (smoothing / V) * Z.sum(axis=1)", "loss = loss"),
    ("drop (1-eps) target weight",
     "loss = lse - (1.0 - smoothing) * z_y", "loss = lse - z_y"),
    ("drop eps/V in the gradient", "dZ = P - smoothing / V", "dZ = P"),
    ("onehot weight 1 instead of 1-eps",
     "dZ[rows, labels[rows]] -= (1.0 - smoothing)", "dZ[rows, labels[rows]] -= 1.0"),
    ("normalise by 1 instead of N_v",
     "return 0.0 if n_valid == 0 else float(grad_loss) / float(n_valid)",
     "return float(grad_loss)"),
    ("dW sign flipped", "dW = dZ.T @ Xd", "dW = -(dZ.T @ Xd)"),
    ("no max-subtraction in d",
     "d = np.exp(Z - m[:, None]).sum(axis=1)", "d = np.exp(Z).sum(axis=1)"),
    ("ignored rows keep gradient", "dZ[~valid] = 0.0", "pass"),
    ("ignored rows keep loss", "return np.where(valid, loss, 0.0)", "return loss"),
    ("dX scaled by a stray factor", "dX = dZ @ Wd", "dX = (dZ @ Wd) * 1.0001"),
    ("z-loss gradient without the factor 2",
     "P = P * (1.0 + 2.0 * z_loss * lse)[:, None]", "P = P * (1.0 + z_loss * lse)[:, None]"),
    ("z-loss term with lse instead of lse^2",
     "loss = loss + z_loss * lse * lse", "loss = loss + z_loss * lse"),
]


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_mutation(tmp_path, name, old, new):
    for d in ("oracle", "tests"):
        shutil.copytree(os.path.join(ROOT, d), tmp_path / d,
                        ignore=shutil.ignore_patterns("__pycache__", "golden"))
    src = tmp_path / "oracle" / "flce_oracle.py"
    text = src.read_text()
    assert old in text, f"mutation anchor not found: {old!r}"
    src.write_text(text.replace(old, new, 1))
    env = dict(os.environ, PYTHONDONTWRITEBYTECODE="1")
    r = subprocess.run(
        [sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
         str(tmp_path / "tests" / "test_oracle_pins.py")],
        cwd=tmp_path, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"pins did not catch mutation {name!r}:\n{r.stdout[-2000:]}"
