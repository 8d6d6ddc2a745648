"""Host-side checks of the C-ABI library: no GPU needed.

The library must load, export every function include/flce.h declares, and plan
workspaces that never hold an N x V logit-shaped buffer.
"""
import ctypes
import json
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "flce.h")


@pytest.fixture(scope="module")
def L():
    from linear_cross_entropy_logit_gb300 import build, binding
    build.build()
    return binding.lib()


def _dz_buffers(B):
    """dZ buffers a backward workspace holds: two with merged launches."""
    return 2 if (B.flce_backward_merge() == 1 and B.flce_cta_pair()) else 1


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b(flce_[a-z_0-9]+)\s*\(", text)
    return sorted(set(names))


def test_header_exports_all(L):
    names = declared_functions()
    assert "flce_forward" in names and "flce_backward" in names and "flce_fwd_bwd" in names
    for n in names:
        assert hasattr(L, n), f"{n} declared in flce.h but not exported"


def test_debug_library_exports_all():
    """The FLCE_DEBUG build exports the same C ABI."""
    from linear_cross_entropy_logit_gb300 import binding as B
    D = B.load(B.DEBUG_LIB_PATH)
    for n in declared_functions():
        assert hasattr(D, n), f"{n} declared in flce.h but not exported by the debug build"
    assert D.flce_abi_version() == 106


def test_status_strings_and_version(L):
    assert L.flce_abi_version() == 106
    for s in range(8):
        assert L.flce_status_string(s).decode().startswith("FLCE_")


def test_workspace_plan_bounded():
    from linear_cross_entropy_logit_gb300 import binding as B
    from linear_cross_entropy_logit_gb300.inputs import CONFIGS
    B.flce_set_vocab_chunk(0)
    for spec in CONFIGS.values():
        if spec.dtype != "bf16":
            continue
        N, H, V = spec.N, spec.H, spec.V
        cv = B.flce_vocab_chunk(N, H, V)
        bufs = _dz_buffers(B)
        assert cv % 256 == 0 and 256 <= cv <= V // (2 * bufs)
        nxv = N * V * 2
        ws = B.flce_workspace_size(N, H, V, B.FLCE_BF16, B.MODE_FWD_BWD)
        # the dZ buffers are the only logit-shaped region: together at most
        # half of N x V and at most the bytes of 1024 rows of logits (or 256 MiB)
        assert bufs * N * cv * 2 <= min(nxv // 2, max(256 << 20, 1024 * V * 2))
        # whole workspace: dZ buffers + fp32 dX accumulator + forward partials
        assert ws <= bufs * N * cv * 2 + N * H * 4 + (40 << 20)
        assert ws < nxv


def test_workspace_matches_pages_fused_figure():
    """The dZ chunk at the worked example of "Fused cross-entropy -- the memory
    kernel" (B*T = 8192, V = 128256, d = 4096) is no larger than one 1024-row
    chunk of logits the page quotes for the fully fused path (0.26 GB)."""
    from linear_cross_entropy_logit_gb300 import binding as B
    figs = json.load(open(os.path.join(ROOT, "tests", "golden", "pages_memory_figures.json")))
    fused = [f for f in figs["figures"] if f["N"] == 1024 and f["V"] == 128256][0]
    B.flce_set_vocab_chunk(0)
    cv = B.flce_vocab_chunk(8192, 4096, 128256)
    assert _dz_buffers(B) * 8192 * cv * 2 / 1e9 <= fused["printed_gb"] + 0.01


def test_workspace_invalid_shapes():
    from linear_cross_entropy_logit_gb300 import binding as B
    assert B.flce_workspace_size(10, 12, 100, B.FLCE_BF16, B.MODE_FWD) == 0  # H % 8
    assert B.flce_workspace_size(-1, 16, 100, B.FLCE_BF16, B.MODE_FWD) == 0
    assert B.flce_workspace_size(10, 16, 0, B.FLCE_BF16, B.MODE_FWD) == 0
    assert B.flce_workspace_size(10, 16, 100, 7, B.MODE_FWD) == 0
    assert B.flce_workspace_size(0, 16, 100, B.FLCE_BF16, B.MODE_FWD_BWD) > 0


def test_backward_merge_setting():
    """Merged backward (opt-in) plans two dZ buffers and a tile counter per
    chunk; off (the default), one buffer of twice the width (same total budget)."""
    from linear_cross_entropy_logit_gb300 import binding as B
    N, H, V = 8192, 4096, 128256
    assert not B.flce_backward_merge()
    B.flce_set_vocab_chunk(0)
    try:
        B.flce_set_backward_merge(True)
        cv2 = B.flce_vocab_chunk(N, H, V)
        ws2 = B.flce_workspace_size(N, H, V, B.FLCE_BF16, B.MODE_BWD)
        B.flce_set_backward_merge(False)
        cv1 = B.flce_vocab_chunk(N, H, V)
        ws1 = B.flce_workspace_size(N, H, V, B.FLCE_BF16, B.MODE_BWD)
        # two buffers of half the budget; one wave-aligned buffer (16384 -> 14592)
        assert (cv1, cv2) == (14592, 8192)
        # the dZ bytes differ by the buffers; the tile counters and the filter
        # masks (sized by Cv) by a few KiB
        assert abs((ws2 - ws1) - N * 2 * (2 * cv2 - cv1)) <= 64 << 10
        B.flce_set_vocab_chunk(2048)
        a = B.flce_workspace_size(N, H, V, B.FLCE_BF16, B.MODE_BWD)
        B.flce_set_backward_merge(True)
        b = B.flce_workspace_size(N, H, V, B.FLCE_BF16, B.MODE_BWD)
        assert b - a >= N * 2048 * 2  # a second dZ buffer at the same Cv
    finally:
        B.flce_set_backward_merge(False)
        B.flce_set_vocab_chunk(0)


def test_default_chunk_fills_the_dw_waves():
    """The budget width is the largest multiple of 512 whose chunk fits
    max(256 MiB, 1024 rows of bf16 logits over V); with one dZ buffer it is then
    narrowed, by at most 1/8, to the width whose dW launch (Cv/256 x H/256
    tiles) best fills its last wave of P = 76 CTA pairs (a 152-SM GB300, also
    the value without a device), unless no narrower width fills it 2.5 points
    better."""
    from linear_cross_entropy_logit_gb300 import binding as B
    B.flce_set_vocab_chunk(0)
    assert B.flce_backward_merge() == 0
    P = 76

    def fill(w, hb):
        tiles = (w // 256) * hb
        return tiles / (-(-tiles // P) * P)

    cases = {  # (N, H, V): (budget width, expected)
        (8192, 4096, 128256): (16384, 14592),   # 57 blocks x 16 = 912 tiles = 12 whole waves
        (16384, 4096, 128256): (8192, 8192),    # 512 tiles fill 96%; 7168 fills 98%, < 2.5 better
        (16384, 3584, 152064): (9216, 8192),    # 504 tiles fill 95%, 448 fill 98%
        (32768, 2304, 256000): (7680, 7680),    # 9 column blocks: multiples of 512; 270 tiles
    }
    for (N, H, V), (budget, want) in cases.items():
        cv = B.flce_vocab_chunk(N, H, V)
        assert cv == want, (N, H, V, cv)
        hb = -(-H // 256)
        assert budget * 7 <= cv * 8 and cv <= budget
        assert cv == budget or fill(cv, hb) > fill(budget, hb) + 0.025
        if hb % 2:
            assert cv % 512 == 0


def test_vocab_chunk_setting():
    from linear_cross_entropy_logit_gb300 import binding as B
    try:
        B.flce_set_vocab_chunk(1000)
        assert B.flce_vocab_chunk(8192, 4096, 128256) == 1024
        B.flce_set_vocab_chunk(10 ** 9)
        bufs = _dz_buffers(B)
        assert B.flce_vocab_chunk(8192, 4096, 128256) == 128256 // (2 * bufs) // 256 * 256
    finally:
        B.flce_set_vocab_chunk(0)


def test_argument_errors_without_gpu(L):
    """Bad arguments are rejected before any CUDA call (so no GPU is needed)."""
    from linear_cross_entropy_logit_gb300 import binding as B
    P = ctypes.c_void_p
    fake = 1 << 20  # aligned non-null addresses; never dereferenced on error
    # H not a multiple of 8
    st = L.flce_forward(P(fake), P(fake), P(fake), 4, 12, 16, -100, 0.0, 0, 0, P(fake), P(fake),
                        P(fake), P(fake), 1 << 20, P(fake), None)
    assert st == B.FLCE_ERR_ARG
    # smoothing outside [0, 1)
    st = L.flce_forward(P(fake), P(fake), P(fake), 4, 16, 16, -100, 1.0, 0, 0, P(fake), P(fake),
                        P(fake), P(fake), 1 << 20, P(fake), None)
    assert st == B.FLCE_ERR_ARG
    # misaligned X
    st = L.flce_forward(P(fake + 2), P(fake), P(fake), 4, 16, 16, -100, 0.0, 0, 0, P(fake),
                        P(fake), P(fake), P(fake), 1 << 20, P(fake), None)
    assert st == B.FLCE_ERR_ARG
    # workspace too small
    st = L.flce_forward(P(fake), P(fake), P(fake), 4, 16, 16, -100, 0.0, 0, 0, P(fake), P(fake),
                        P(fake), P(fake), 16, P(fake), None)
    assert st == B.FLCE_ERR_WORKSPACE
    # missing err_word
    st = L.flce_fwd_bwd(P(fake), P(fake), P(fake), 4, 16, 16, -100, 0.0, 0, 0, None, P(fake),
                        P(fake), P(fake), P(fake), P(fake), 0, P(fake), 1 << 20, None, None)
    assert st == B.FLCE_ERR_ARG


def test_options_struct_layout(L):
    """The ctypes mirror of flce_options has the C struct's size and defaults."""
    from linear_cross_entropy_logit_gb300 import binding as B
    o = B.FlceOptions()
    L.flce_options_init(ctypes.byref(o))
    assert o.struct_size == ctypes.sizeof(B.FlceOptions)
    assert (o.ignore_index, o.smoothing, o.z_loss, o.reduction, o.row_loss) == (-100, 0.0, 0.0, 0, None)
    assert (o.skip_ignored_blocks, o.grad_filter) == (0, 0.0)
    assert (o.cta_pair, o.backward_merge, o.l2_hints, o.vocab_chunk,
            o.cluster_multicast) == (-1, -1, -1, -1, -1)
    # a struct of another size is rejected before any CUDA call
    o.struct_size = 8
    P = ctypes.c_void_p
    fake = 1 << 20
    st = L.flce_forward_ex(P(fake), P(fake), P(fake), 4, 16, 16, 0, ctypes.byref(o), P(fake),
                           P(fake), P(fake), P(fake), 1 << 20, P(fake), None)
    assert st == B.FLCE_ERR_ARG


def test_plain_c_caller(L, tmp_path):
    """include/flce.h is a C header: a C99 program compiles against it with
    -pedantic, links against libflce.so and gets the same answers as the
    Python binding from the host-only entry points."""
    import shutil
    import subprocess
    from linear_cross_entropy_logit_gb300 import binding as B
    from linear_cross_entropy_logit_gb300 import build as libbuild
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "caller.c"
    src.write_text(
        '#include <stdio.h>\n'
        '#include "flce.h"\n'
        'int main(void) {\n'
        '  flce_options o;\n'
        '  flce_options_init(&o);\n'
        '  printf("%d %lld %zu %lld %s\\n", flce_abi_version(), (long long)o.ignore_index,\n'
        '         flce_workspace_size(8192, 4096, 128256, FLCE_BF16, FLCE_MODE_FWD_BWD),\n'
        '         (long long)flce_vocab_chunk(8192, 4096, 128256),\n'
        '         flce_status_string(FLCE_ERR_ARG));\n'
        '  return 0;\n'
        '}\n')
    exe = tmp_path / "caller"
    libdir = os.path.dirname(libbuild.LIB)
    subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I",
                    os.path.join(ROOT, "include"), str(src), "-L", libdir, "-lflce",
                    f"-Wl,-rpath,{libdir}", "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()
    assert int(out[0]) == L.flce_abi_version()
    assert int(out[1]) == -100
    assert int(out[2]) == B.flce_workspace_size(8192, 4096, 128256, B.FLCE_BF16, B.MODE_FWD_BWD)
    assert int(out[3]) == B.flce_vocab_chunk(8192, 4096, 128256)
    assert out[4].startswith("FLCE_ERR_ARG")


def test_options_launch_settings_size_the_workspace(L):
    """Launch settings in flce_options override the process-wide defaults for
    one call, and flce_workspace_size_ex sizes with them; -1 fields and a
    struct of the 1.05 size (no such fields) take the defaults."""
    from linear_cross_entropy_logit_gb300 import binding as B
    N, H, V = 8192, 4096, 128256
    B.flce_set_vocab_chunk(0)
    B.flce_set_backward_merge(False)
    B.flce_set_cta_pair(True)
    base = B.flce_workspace_size(N, H, V, B.FLCE_BF16, B.MODE_BWD)
    o = B.make_options()
    assert B.flce_workspace_size(N, H, V, B.FLCE_BF16, B.MODE_BWD, o) == base
    assert B.flce_vocab_chunk(N, H, V, o) == 14592
    merged = B.make_options(backward_merge=True)
    assert B.flce_vocab_chunk(N, H, V, merged) == 8192
    try:
        B.flce_set_backward_merge(True)
        assert B.flce_workspace_size(N, H, V, B.FLCE_BF16, B.MODE_BWD, merged) == \
            B.flce_workspace_size(N, H, V, B.FLCE_BF16, B.MODE_BWD)
        # an explicit 0 ignores the process-wide 1
        off = B.make_options(backward_merge=False)
        assert B.flce_workspace_size(N, H, V, B.FLCE_BF16, B.MODE_BWD, off) == base
    finally:
        B.flce_set_backward_merge(False)
    chunk = B.make_options(vocab_chunk=2048)
    assert B.flce_vocab_chunk(N, H, V, chunk) == 2048
    assert B.flce_vocab_chunk(N, H, V) == 14592
    # the 1.05 struct (no launch settings) is accepted and takes the defaults
    old = B.make_options(vocab_chunk=2048)
    old.struct_size = B.FlceOptions.cta_pair.offset
    assert B.flce_workspace_size(N, H, V, B.FLCE_BF16, B.MODE_BWD, old) == base
    # out-of-range settings are rejected (size 0)
    for field, bad in (("cta_pair", 2), ("backward_merge", -2), ("l2_hints", 3),
                       ("vocab_chunk", -5), ("cluster_multicast", 2)):
        o = B.make_options()
        setattr(o, field, bad)
        assert B.flce_workspace_size(N, H, V, B.FLCE_BF16, B.MODE_BWD, o) == 0, field


def test_options_sizing_is_thread_safe():
    """Two threads size workspaces with their own launch settings while a
    third keeps flipping the process-wide defaults: each thread's sizes never
    change, so a workspace sized this way always fits its call."""
    import threading
    from linear_cross_entropy_logit_gb300 import binding as B
    N, H, V = 8192, 4096, 128256
    mine = {"merged": B.make_options(backward_merge=True, cta_pair=True, vocab_chunk=0),
            "plain": B.make_options(backward_merge=False, cta_pair=False, vocab_chunk=4096)}
    want = {k: B.flce_workspace_size(N, H, V, B.FLCE_BF16, B.MODE_FWD_BWD, o)
            for k, o in mine.items()}
    assert want["merged"] != want["plain"]
    stop = threading.Event()
    bad = []

    def flipper():
        i = 0
        while not stop.is_set():
            B.flce_set_backward_merge(i % 2 == 0)
            B.flce_set_cta_pair(i % 3 != 0)
            B.flce_set_vocab_chunk((i % 4) * 1024)
            i += 1

    def sizer(key):
        for _ in range(3000):
            got = B.flce_workspace_size(N, H, V, B.FLCE_BF16, B.MODE_FWD_BWD, mine[key])
            if got != want[key]:
                bad.append((key, got))
                return

    t0 = threading.Thread(target=flipper)
    ts = [threading.Thread(target=sizer, args=(k,)) for k in mine]
    t0.start()
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    stop.set()
    t0.join()
    B.flce_set_backward_merge(False)
    B.flce_set_cta_pair(True)
    B.flce_set_vocab_chunk(0)
    assert not bad


def test_noalloc_rejects_misaligned_words(L):
    """flce_forward_noalloc refuses 32-bit outputs that are not 4-byte aligned
    on the host, before any CUDA call (no GPU needed)."""
    from linear_cross_entropy_logit_gb300 import binding as B
    P = ctypes.c_void_p
    fake = 1 << 20
    args = [P(fake), P(fake), P(fake), 64, 64, 1000, -100, 0.0, 0]
    outs = [P(fake), P(fake), P(fake), P(fake)]  # loss, lse, valid_count, err_word
    for i in range(4):
        o = list(outs)
        o[i] = P(fake + 2)
        assert L.flce_forward_noalloc(*args, *o, None) == B.FLCE_ERR_ARG, i
