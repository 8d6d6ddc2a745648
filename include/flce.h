/*
 * flce.h -- fused linear cross-entropy on one GB300 (sm_103a): C ABI.
 *
 * The library computes, for hidden states X (N x H), an unembedding matrix W
 * (V x H) and integer targets y (N):
 *
 *   Z      = X W^T                       logits, never stored (N x V)
 *   lse_i  = m_i + log sum_j exp(z_ij - m_i),  m_i = max_j z_ij
 *   l_i    = valid_i * (lse_i - (1-eps) z_{i,y_i} - (eps/V) sum_j z_ij)
 *   loss   = sum_i l_i / N_valid  (mean)   or   sum_i l_i  (sum)
 *   dZ_ij  = c * valid_i * (exp(z_ij - lse_i) - (1-eps) 1[j = y_i] - eps/V)
 *   dX     = dZ W,   dW = dZ^T X  (dW += when accumulating)
 *
 * with valid_i = (y_i != ignore_index), N_valid = sum_i valid_i and
 * c = grad_loss / N_valid (mean; 0 when N_valid = 0) or c = grad_loss (sum).
 *
 * Sources (page title, section):
 *   "Chunked and Fused Cross-Entropy: How Online Logit Tiling Slashes
 *    Large-Vocabulary VRAM Bottlenecks in LLM Training" -- the projection and
 *    loss equations ("The Vocabulary Memory Wall in Modern LLMs") and steps
 *    1-4 of "Mathematical Mechanics of Chunked Online Cross-Entropy"; label
 *    -100 masking and label smoothing ("Numerical Considerations and
 *    Practical Trade-Offs", items 2-3).
 *   "Cut Cross-Entropy: Memory-Efficient Large-Vocab LLM Guide" -- the call
 *    linear_cross_entropy(h, W, labels, ignore_index=-100) and the chunked
 *    reference's mean over max(valid_token_count, 1).
 *   "Fused cross-entropy -- the memory kernel" -- dlogits = (p - y)/N,
 *    "Trick 1" (online softmax) and "Trick 2" (fuse the lm-head matmul).
 * Label smoothing follows PyTorch's convention (eps/V of the mass on every
 * class, the target keeps 1 - eps + eps/V); the pages name the term without
 * a formula.
 *
 * Conventions for every entry point
 *   - All tensor pointers are DEVICE pointers, row-major and contiguous:
 *     X is N x H, W is V x H (the nn.Linear weight layout), labels is N int64,
 *     dX is N x H, dW is V x H float32, lse is N float32.
 *   - X, W and dX use `dtype` (bf16 or fp32); X, W, dX, dW must be 16-byte
 *     aligned and H must be a multiple of 8 (rows are fetched by TMA).
 *   - fp32 inputs are rounded to bf16 once (in the workspace) and multiplied
 *     on the bf16 tensor cores with fp32 accumulation; dX is then fp32.
 *   - The caller owns every buffer, the workspace included.  The library
 *     allocates no device memory and never materialises an N x V tensor: its
 *     largest region is an N x Cv bf16 gradient chunk with Cv <= V/2.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL is the legacy
 *     default stream) and never synchronise the host.
 *   - Argument errors are reported synchronously by the return value and
 *     launch nothing.  Data errors are reported through *err_word (device
 *     int32 the caller zeroes beforehand; the first error code wins and stays
 *     set): FLCE_ERR_LABEL for a label outside [0, V) that is not
 *     ignore_index (that row then counts as ignored), FLCE_ERR_TIMEOUT if a
 *     kernel's bounded wait expired (outputs are then undefined).  Read it
 *     after synchronising the stream.
 *   - N = 0 is allowed (loss 0, no valid tokens, dW zeroed unless
 *     accumulating).  ignore_index may be any value; a value inside [0, V)
 *     masks that class.
 */
#ifndef FLCE_H_
#define FLCE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FLCE_OK = 0,
  FLCE_ERR_ARG = 1,          /* bad pointer, size, alignment or option      */
  FLCE_ERR_UNSUPPORTED = 2,  /* no sm_100-family device, or a size limit     */
  FLCE_ERR_WORKSPACE = 3,    /* workspace missing or smaller than required  */
  FLCE_ERR_LABEL = 4,        /* (err_word only) label outside [0, V)        */
  FLCE_ERR_TIMEOUT = 5,      /* (err_word only) a bounded device wait expired */
  FLCE_ERR_CUDA = 6,         /* a CUDA runtime/driver call failed           */
  FLCE_ERR_BOUNDS = 7        /* (err_word only, debug build) an index check
                                failed; the access was skipped              */
} flce_status;

typedef enum { FLCE_BF16 = 0, FLCE_FP32 = 1 } flce_dtype;
typedef enum { FLCE_MEAN = 0, FLCE_SUM = 1 } flce_reduction;
typedef enum { FLCE_MODE_FWD = 1, FLCE_MODE_BWD = 2, FLCE_MODE_FWD_BWD = 3 } flce_mode;

/* Bytes of workspace one call of `mode` needs for this shape (0 on invalid
 * arguments).  Pure host arithmetic: needs no GPU.  The layout depends only on
 * (N, H, V, dtype, mode) and the launch settings -- the vocabulary chunk
 * width, merged backward launches and the tile shape.  This form reads the
 * process-wide settings below at the time of the call; flce_workspace_size_ex
 * (after flce_options) takes them from an options struct, so that sizing and
 * the call that uses the workspace cannot disagree when another thread changes
 * a process-wide setting in between. */
size_t flce_workspace_size(int64_t N, int64_t H, int64_t V, flce_dtype dtype, int mode);

/* Vocabulary columns per backward chunk (Cv): the gradient scratch is N x Cv
 * bf16, two such buffers when the merged backward below is enabled.  0 (the
 * default) picks the largest multiple of 512 whose buffers together fit in
 * max(256 MiB, 1024 * V * 2 bytes) -- the bytes of 1024 token rows of bf16
 * logits, the fully fused chunk of "Fused cross-entropy -- the memory
 * kernel" -- clamped to [256, V/2] (one buffer) or [256, V/4] (two buffers);
 * with one buffer it is then narrowed, by at most 1/8, to the width whose
 * weight-gradient launch ((Cv / 256) * ceil(H / 256) tiles) best fills its
 * last wave of the current device's CTA pairs (a multiple of 512 when
 * ceil(H / 256) is odd).  A set value is rounded up to a multiple of 256 and
 * clamped the same way.  Process-wide default of the calls whose options leave
 * vocab_chunk at -1 (the plain calls always use it); set it before sizing
 * workspaces.  flce_vocab_chunk returns the width such a call of this shape
 * uses (0 on invalid arguments). */
flce_status flce_set_vocab_chunk(int64_t cols);
int64_t flce_vocab_chunk(int64_t N, int64_t H, int64_t V);

/* GEMM tile shape, process-wide default (options field cta_pair overrides it
 * per call).  1 (the default): a cluster of two CTAs on two SMs computes each
 * 256 x 256 tile with tcgen05.mma.cta_group::2, each CTA loading its own 128
 * rows of A and half of B.  0: one CTA per 128 x 256 tile.  Both give the
 * same results up to fp32 summation order. */
flce_status flce_set_cta_pair(int on);
int flce_cta_pair(void);

/* Operand multicast between CTA pairs, process-wide default (options field
 * cluster_multicast overrides it per call).  1 (the default): a CTA-pair GEMM
 * launch of the plain kernels (none of skip_ignored_blocks, grad_filter, L2
 * hints) whose tiles pair up -- an even number of row blocks sharing each
 * column block, or of column blocks sharing each row block -- is launched
 * with 4-CTA clusters preferred; the two pairs of a 4-CTA cluster compute two
 * such tiles in step and multicast the operand they share (TMA .multicast),
 * so each loads a quarter less from L2.  The hardware may group any four CTAs
 * as two 2-CTA clusters instead; those compute the same tiles without
 * multicast.  0: plain CTA pairs.  Results are bit-identical either way.
 * Not used by the merged backward launches. */
flce_status flce_set_cluster_multicast(int on);
int flce_cluster_multicast(void);

/* Backward layout, process-wide default (options field backward_merge
 * overrides it per call).  With CTA-pair tiles and none of the optional
 * features (skip_ignored_blocks, grad_filter, L2 hints):
 *   0 (the default): per vocabulary chunk three launches -- the dZ
 *     recompute, the dW GEMM, the dX GEMM -- and one dZ buffer;
 *   1: the dZ recompute of chunk 0 alone, then one launch per chunk c holding
 *     the dW and dX GEMMs of c and the dZ recompute of c+1 in one tile list,
 *     so no GEMM ends on its own partial wave; the workspace then holds two
 *     N x Cv dZ buffers;
 *   2: per chunk the dZ recompute alone, then one launch of the dW and dX
 *     GEMMs of that chunk from one tile list (one dZ buffer).
 * Layouts 1 and 2 add one int per chunk to the workspace.  All give
 * bit-identical results for the same Cv.  Layout 1 pays when Cv is small
 * next to the tile grid (measured on a GB300 at the Llama-3 shape: 6.8%
 * faster steps at Cv = 2048, 2.5% at 4096); at the default chunk width, and
 * at equal dZ memory, the three-launch backward was as fast or faster.  Set
 * it before sizing workspaces; other values return FLCE_ERR_ARG. */
flce_status flce_set_backward_merge(int on);
int flce_backward_merge(void);

/* L2 residency hints, process-wide default (options field l2_hints overrides
 * it per call).  1: the operand a GEMM re-reads on every
 * wave of tiles (X, or a W chunk) is loaded with an evict_last policy covering
 * up to ~64 MB of L2.  0 (the default; on a GB300 the hints did not speed up
 * the llama3-shaped step and slowed the dW GEMM by ~3%): no hints.  Results do
 * not depend on it. */
flce_status flce_set_l2_hints(int on);

/* Forward ("Mathematical Mechanics of Chunked Online Cross-Entropy", steps
 * 1-2): loss (device float, 1), lse (device float, N, every row including
 * ignored ones), valid_count (device int32, 1: N_valid).  workspace: device,
 * 256-byte aligned, at least flce_workspace_size(..., FLCE_MODE_FWD). */
flce_status flce_forward(const void* X, const void* W, const int64_t* labels, int64_t N,
                         int64_t H, int64_t V, int64_t ignore_index, float smoothing,
                         flce_dtype dtype, flce_reduction reduction, float* loss, float* lse,
                         int32_t* valid_count, void* workspace, size_t ws_bytes,
                         int32_t* err_word, void* stream);

/* Backward (steps 3-4): recomputes the logits tile by tile from X, W and the
 * forward's lse, forms dZ in bf16 and writes dX (N x H, dtype, overwritten)
 * and dW (V x H fp32; overwritten, or added to when accumulate_dW != 0).
 * valid_count: the forward's N_valid (device int32) -- a data-parallel caller
 * may pass the global count.  grad_loss: device float (upstream gradient of
 * the loss) or NULL for 1.  workspace: >= flce_workspace_size(..., FLCE_MODE_BWD). */
flce_status flce_backward(const void* X, const void* W, const int64_t* labels, int64_t N,
                          int64_t H, int64_t V, int64_t ignore_index, float smoothing,
                          flce_dtype dtype, flce_reduction reduction, const float* lse,
                          const int32_t* valid_count, const float* grad_loss, void* dX,
                          float* dW, int accumulate_dW, void* workspace, size_t ws_bytes,
                          int32_t* err_word, void* stream);

/* Forward then backward in one call (the fused training step of the pages'
 * "Trick 2"): loss, lse, valid_count, dX, dW as above.
 * workspace: >= flce_workspace_size(..., FLCE_MODE_FWD_BWD). */
flce_status flce_fwd_bwd(const void* X, const void* W, const int64_t* labels, int64_t N,
                         int64_t H, int64_t V, int64_t ignore_index, float smoothing,
                         flce_dtype dtype, flce_reduction reduction, const float* grad_loss,
                         float* loss, float* lse, int32_t* valid_count, void* dX, float* dW,
                         int accumulate_dW, void* workspace, size_t ws_bytes, int32_t* err_word,
                         void* stream);

/* Options of the extended entry points: z-loss, a per-token loss output and
 * skipping of fully ignored token blocks (instruction tuning), besides the
 * options of the plain calls.  Initialise with
 * flce_options_init, then set fields:
 *   ignore_index  labels equal to it are masked (default -100)
 *   smoothing     label smoothing eps in [0, 1) (default 0)
 *   z_loss        z-loss weight alpha >= 0 (default 0): each valid token adds
 *                 alpha * lse_i^2 to its loss ("Chunked and Fused
 *                 Cross-Entropy ...", "Numerical Considerations and Practical
 *                 Trade-Offs", item 3: L_z = alpha log^2 sum exp(z)); averaged
 *                 like the cross-entropy; the gradient gains
 *                 c * 2 alpha lse_i * softmax_ij
 *   reduction     FLCE_MEAN or FLCE_SUM (default FLCE_MEAN)
 *   row_loss      NULL, or a device float[N] that receives every token's loss
 *                 l_i (0 on ignored rows): the per-token ("none") reduction.
 *   skip_ignored_blocks
 *                 0 (default) or 1: skip the projection and the backward GEMMs
 *                 for blocks of 256 consecutive tokens (128 with
 *                 flce_set_cta_pair(0)) whose labels are all ignore_index --
 *                 instruction tuning masks whole prompt spans ("Chunked and
 *                 Fused Cross-Entropy ...", "Numerical Considerations ...",
 *                 item 2).  loss, dX and dW are unchanged; lse of the rows of a
 *                 skipped block is NaN.
 *   grad_filter   0 (default) or a threshold eps_f in (0, 1), e.g. 2^-12:
 *                 gradient filtering after Cut Cross-Entropy ("Chunked and
 *                 Fused Cross-Entropy ...", "Apple Cut Cross-Entropy (CCE)"):
 *                 the dX and dW GEMMs skip every 32-token x 64-column block of
 *                 dZ whose probabilities are all below eps_f and that holds no
 *                 target.  An approximation: the dropped entries each have
 *                 |dZ| <= c * max((1 + 2 alpha lse) eps_f, eps / V), so
 *                 |delta dX|_F <= |delta dZ|_F |W|_2 and |delta dW|_F <=
 *                 |delta dZ|_F |X|_2.  Needs ceil(Cv/64) and ceil(N/64) <= 1024
 *                 (else FLCE_ERR_UNSUPPORTED); loss and lse are exact.
 * Launch settings of this call (ABI 1.06; flce_options_init sets each to -1,
 * which takes the process-wide setting of the matching flce_set_* call at
 * the time of the call; any other value holds for this call only, so callers
 * in several threads can use different settings without racing):
 *   cta_pair        -1, 0 or 1: see flce_set_cta_pair
 *   backward_merge  -1, 0, 1 or 2: see flce_set_backward_merge
 *   l2_hints        -1, 0 or 1: see flce_set_l2_hints
 *   vocab_chunk     -1, 0 (automatic width) or a width in columns: see
 *                   flce_set_vocab_chunk
 *   cluster_multicast -1, 0 or 1: see flce_set_cluster_multicast
 * The workspace of a call must be sized with the same settings:
 * flce_workspace_size_ex with the same options.  A struct from a caller built
 * against ABI 1.05 (struct_size = offsetof(flce_options, cta_pair)) is
 * accepted and runs with the process-wide settings. */
typedef struct flce_options {
  size_t struct_size;
  int64_t ignore_index;
  float smoothing;
  float z_loss;
  flce_reduction reduction;
  float* row_loss;
  int skip_ignored_blocks;
  float grad_filter;
  int cta_pair;
  int backward_merge;
  int l2_hints;
  int64_t vocab_chunk;
  int cluster_multicast;
} flce_options;

void flce_options_init(flce_options* opt);

/* flce_workspace_size / flce_vocab_chunk for a call made with these options
 * (NULL: the process-wide settings).  0 on invalid arguments or options. */
size_t flce_workspace_size_ex(int64_t N, int64_t H, int64_t V, flce_dtype dtype, int mode,
                              const flce_options* opt);
int64_t flce_vocab_chunk_ex(int64_t N, int64_t H, int64_t V, const flce_options* opt);

flce_status flce_forward_ex(const void* X, const void* W, const int64_t* labels, int64_t N,
                            int64_t H, int64_t V, flce_dtype dtype, const flce_options* opt,
                            float* loss, float* lse, int32_t* valid_count, void* workspace,
                            size_t ws_bytes, int32_t* err_word, void* stream);

flce_status flce_backward_ex(const void* X, const void* W, const int64_t* labels, int64_t N,
                             int64_t H, int64_t V, flce_dtype dtype, const flce_options* opt,
                             const float* lse, const int32_t* valid_count,
                             const float* grad_loss, void* dX, float* dW, int accumulate_dW,
                             void* workspace, size_t ws_bytes, int32_t* err_word, void* stream);

flce_status flce_fwd_bwd_ex(const void* X, const void* W, const int64_t* labels, int64_t N,
                            int64_t H, int64_t V, flce_dtype dtype, const flce_options* opt,
                            const float* grad_loss, float* loss, float* lse,
                            int32_t* valid_count, void* dX, float* dW, int accumulate_dW,
                            void* workspace, size_t ws_bytes, int32_t* err_word, void* stream);

/* Vocabulary-parallel layout (the "tiled vocabulary dot
 * products" of "Chunked and Fused Cross-Entropy ...", comparison table, with
 * step 2's running (m, d) carried across vocabulary shards).  Shard p holds
 * rows [vocab_offset, vocab_offset + V_shard) of W for a vocabulary of
 * vocab_total; labels stay global.  A step is:
 *   1. every shard: flce_forward_vocab_shard -> partials (device float[N][4]:
 *      max * log2(e), sum of exp(z - max) rescaled, the target logit if the
 *      label is in this shard else 0, the shard's row sum of logits);
 *   2. gather the P shards' partials into one device float[P][N][4] (the
 *      exchange, e.g. an all-gather of N * 16 bytes per shard) and call
 *      flce_combine_vocab_shards -> loss, lse, valid_count (the LSE-combine);
 *   3. every shard: flce_backward_vocab_shard with the global lse and
 *      valid_count -> its fp32 partial dX (N x H; the shards' partials sum to
 *      dX: an all-reduce) and its own dW rows (V_shard x H fp32).
 * opt: ignore_index, smoothing (eps / vocab_total per class), z_loss,
 * reduction and the launch settings; row_loss only in the combine;
 * skip_ignored_blocks must be 0.  Workspaces: flce_workspace_size_ex(N, H,
 * V_shard, dtype, FLCE_MODE_FWD / _BWD, opt) for the shard calls,
 * flce_combine_workspace_size(N) for the combine. */
flce_status flce_forward_vocab_shard(const void* X, const void* W_shard, const int64_t* labels,
                                     int64_t N, int64_t H, int64_t V_shard, int64_t vocab_offset,
                                     int64_t vocab_total, flce_dtype dtype,
                                     const flce_options* opt, float* partials, void* workspace,
                                     size_t ws_bytes, int32_t* err_word, void* stream);

size_t flce_combine_workspace_size(int64_t N);

flce_status flce_combine_vocab_shards(const float* partials, int n_shards, int64_t N,
                                      const int64_t* labels, int64_t vocab_total,
                                      const flce_options* opt, float* loss, float* lse,
                                      int32_t* valid_count, void* workspace, size_t ws_bytes,
                                      int32_t* err_word, void* stream);

flce_status flce_backward_vocab_shard(const void* X, const void* W_shard, const int64_t* labels,
                                      int64_t N, int64_t H, int64_t V_shard,
                                      int64_t vocab_offset, int64_t vocab_total,
                                      flce_dtype dtype, const flce_options* opt,
                                      const float* lse, const int32_t* valid_count,
                                      const float* grad_loss, float* dX_partial,
                                      float* dW_shard, int accumulate_dW, void* workspace,
                                      size_t ws_bytes, int32_t* err_word, void* stream);

/* Human-readable name of a status code (static string). */
const char* flce_status_string(flce_status s);

/* Text of the last CUDA error this thread saw inside the library ("" if none). */
const char* flce_last_cuda_error(void);

/* Number of kernels the last flce_forward / flce_backward / flce_fwd_bwd call
 * on this thread enqueued. */
int flce_last_launch_count(void);

/* Optional per-kernel timing.  While enabled (per host thread), every GEMM
 * launch of the calls above is bracketed by two CUDA events recorded on the
 * caller's stream.  flce_profile_read synchronises the recorded events and
 * returns the accumulated device time and launch count of one kernel kind:
 * 0 forward logits + online LSE, 1 dZ recompute, 2 dW GEMM, 3 dX GEMM,
 * 4 merged backward launch (dW and dX of one chunk, dZ of the next).
 * flce_profile_reset clears the totals. */
flce_status flce_profile_enable(int on);
flce_status flce_profile_read(int kind, double* total_ms, int* launches);
void flce_profile_reset(void);

/* Forward without any allocation and without a workspace argument.
 * The pages have no counterpart to this entry point: it exists for callers
 * that cannot call cudaMalloc or keep a workspace -- code inside a host
 * application that owns all device memory through its own fixed pool, code
 * on a path that must not allocate after start-up, and C callers without an
 * allocator.  Outputs as flce_forward's (loss, lse, valid_count, err_word);
 * the values match flce_forward's within the parity tolerances, not bit for
 * bit: this entry point always runs the 128 x 256 single-CTA tiles with its
 * own vocabulary grouping, so its sums run in another order.  bf16 X and W
 * only.  err_word, loss, valid_count and lse must be 4-byte aligned.
 * loss and lse are undefined whenever *err_word is FLCE_ERR_TIMEOUT after
 * the call: the merge may then have read partials an earlier call left in
 * the shared scratch.
 * Scratch: a fixed device array of FLCE_NOALLOC_SCRATCH_BYTES inside the
 * library, held on every GPU that runs this entry point until the process
 * exits.  The first call on a device looks up the array's address (make that
 * call before any stream capture).  Shapes whose forward partials do not fit
 * return FLCE_ERR_WORKSPACE (N up to about 1,000,000 tokens fits).  All calls
 * share the array, so calls whose kernels overlap on the GPU (other streams
 * or host threads) race: serialise them. */
#define FLCE_NOALLOC_SCRATCH_BYTES (16u << 20)
flce_status flce_forward_noalloc(const void* X, const void* W, const int64_t* labels, int64_t N,
                                 int64_t H, int64_t V, int64_t ignore_index, float smoothing,
                                 flce_reduction reduction, float* loss, float* lse,
                                 int32_t* valid_count, int32_t* err_word, void* stream);

/* Text of the last error flce_forward_noalloc met on this thread ("" if none). */
const char* flce_noalloc_last_error(void);

/* ABI version of this header (major * 100 + minor). */
int flce_abi_version(void);

/* TEST-ONLY: runs the library's bounded mbarrier wait (the one every pipeline
 * wait of the GEMM kernels uses) on a barrier nothing arrives on, with a limit
 * of timeout_ns (<= 10 s).  The kernel records FLCE_ERR_TIMEOUT in *err_word,
 * writes the microseconds it waited to *waited_us (device int32) and returns,
 * leaving the CUDA context usable. */
flce_status flce_debug_wait_timeout(int32_t* err_word, uint64_t timeout_ns, int32_t* waited_us,
                                    void* stream);

/* TEST-ONLY: how many GEMM launches of the last call on this thread were made
 * with 4-CTA clusters preferred (the operand-multicast walk of
 * flce_set_cluster_multicast). */
int flce_debug_last_multicast_launches(void);

/* TEST-ONLY: the library's tcgen05 GEMM core without a loss epilogue.
 * D (M x Nn fp32, device, row-major) = A * B^T, or += when accumulate != 0,
 * where A is M x K (a_mn = 0: stored M x K row-major) or stored K x M
 * (a_mn = 1), and B is Nn x K (b_mn = 0: stored Nn x K) or stored K x Nn
 * (b_mn = 1); A and B are bf16.  Exercises the K-major and MN-major operand
 * descriptors in isolation; no part of the loss path calls it. */
flce_status flce_debug_gemm(const void* A, const void* B, float* D, int64_t M, int64_t Nn,
                            int64_t K, int a_mn, int b_mn, int accumulate, int32_t* err_word,
                            void* stream);

#ifdef __cplusplus
}
#endif
#endif /* FLCE_H_ */
