/*
 * csa.h -- C ABI of the GB300 (sm_103a) causal-attention-score library,
 * libcsa_gb300.so.
 *
 * Two products, each a persistent tcgen05/TMA kernel (plus, for dense rows no
 * tensor map can describe, one realigning copy into caller workspace launched
 * before it), and the calls built on them: the batched NT product
 * (batch_matmul_nt), the fused
 * causal softmax of the scores (causal_softmax_forward), the score product
 * over fp32 inputs (trimul_forward_f32), many dense layers sharing W in one
 * launch (dense_xwt_grouped), and an allocation-free score entry point
 * (trimul_forward_noalloc). Each is documented at its declaration below.
 *
 *  trimul_forward  the causal triangular score product of
 *                  "llm.c dev/cuda/trimat_forward.cu" (the CPU referee
 *                  trimul_cpu, Chapter I; the lower-tile skip of trimul_global,
 *                  Chapter II):
 *                    out[b][h][t][t2] = (Q[b][h][t][:] . K[b][h][t2][:]) / sqrt(HS)
 *                                       for t2 <= t, the mask value for t2 > t,
 *                  with Q[b][h][t][d] = qkv[b][t][0][h][d] and
 *                       K[b][h][t2][d] = qkv[b][t2][1][h][d].
 *
 *  dense_xwt       the dense layer of "DietCode tests/codegen/
 *                  test_1_local_padding.py" (test_local_padding docstring):
 *                    Y[i][j] = sum_k X[i][k] * W[j][k]   (Y = X W^T)
 *                  for any M, I, H >= 1; tails are handled only where data is
 *                  fetched (zero fill) and written back (clipped), never in the
 *                  compute stage ("local padding").
 *
 * Conventions shared by every entry point:
 *  - Pointers named as device pointers must point to memory of the current CUDA
 *    device (cudaMalloc'd or torch-allocated). The caller owns every buffer,
 *    scratch space included (dense_xwt_ws); no call allocates device memory.
 *    The library keeps, per device, only fixed arrays in its own image: the
 *    status word, the kernels' work-list counters and the scratch of
 *    trimul_forward_noalloc (plus the page-locked completion words below).
 *  - bf16 inputs are passed as `const void*` to raw 16-bit bfloat16 values.
 *  - Outputs are fp32 and fully overwritten (no read-modify-write).
 *  - `stream` is a cudaStream_t passed as void*; NULL is the legacy default
 *    stream. Calls are asynchronous on that stream; argument errors are
 *    returned synchronously before anything is launched.
 *  - Return value: CSA_OK (0) or a negative csa_status. A failed call launches
 *    nothing and leaves the output untouched; csa_last_error() then describes it.
 *  - Work-list counters (trimul_forward, trimul_forward_ex, trimul_forward_f32,
 *    causal_softmax_forward): these kernels take work from a set of counters
 *    that their last CTA resets. A launch outside stream capture uses its
 *    stream's set (launches on one stream run in order); a stream gets a set
 *    that was never used or whose last launch has reported completion (through
 *    a 2 KB page-locked host array per kernel and device, made at the first such
 *    launch on that device -- make it outside any stream capture). With launches
 *    still in flight on 256 other streams, the call returns CSA_ERR_BUSY. A
 *    launch captured into a CUDA graph gets a set of its own for good, at most
 *    1024 per kernel and process (then CSA_ERR_BUSY); a graph instantiated more
 *    than once must not have two instances running at once. Launches whose work
 *    is dealt statically (lower-only scores, batch_matmul_nt) use no set.
 *  - The library keeps one device status word per device. A kernel whose
 *    bounded wait ran out records CSA_ERR_TIMEOUT there and returns early
 *    (its output is then incomplete); csa_get_status() reports and clears it.
 *  - Thread safety: entry points may be called from several host threads; the
 *    error string is per thread. Each call works on the calling thread's current
 *    device (cudaGetDevice); the first call on a thread makes that device's
 *    primary context current there (cudaSetDevice).
 */
#ifndef CSA_GB300_H
#define CSA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int csa_status;

#define CSA_OK                 0
#define CSA_ERR_NULL          -1  /* a required pointer is NULL */
#define CSA_ERR_SHAPE         -2  /* a size is <= 0, C % NH != 0, or an index overflows */
#define CSA_ERR_ALIGN         -3  /* a pointer or stride breaks the 16-byte rule below */
#define CSA_ERR_UNSUPPORTED   -4  /* a size beyond what the kernel implements (HS > 256) */
#define CSA_ERR_ARCH          -5  /* the current device is not sm_103 (GB300) */
#define CSA_ERR_LAUNCH        -6  /* the kernel launch failed (see csa_last_error) */
#define CSA_ERR_TIMEOUT       -7  /* a device-side bounded wait ran out (csa_get_status) */
#define CSA_ERR_CUDA          -8  /* a CUDA runtime/driver call failed (no device, ...) */
#define CSA_ERR_CHECK         -9  /* a device-side index check of a debug build (built with
                                     -DCSA_DEBUG) failed (reported by csa_get_status) */
#define CSA_ERR_WORKSPACE    -10  /* dense_xwt_ws: workspace missing or smaller than
                                     dense_xwt_workspace_size reports */
#define CSA_ERR_BUSY         -11  /* no work-list counter set free: score or softmax
                                     launches in flight on 256 other streams, or more
                                     than 1024 of them captured into CUDA graphs */

/* Causal mask bit patterns for the upper triangle (t2 > t). The page writes
 * NAN (the float quiet NaN, 0x7FC00000) and notes -inf would also do. */
#define CSA_MASK_NAN          0x7FC00000u
#define CSA_MASK_NEG_INF      0xFF800000u

/* trimul_forward_ex flags. */
#define CSA_TRIMUL_FULL        0u  /* write every element: scores below, mask above */
#define CSA_TRIMUL_LOWER_ONLY  1u  /* write only t2 <= t; leave t2 > t untouched
                                      (what the page's GPU kernels do, tri4's
                                      "don't write above the diagonal") */

/*
 * trimul_forward -- causal score product, NaN mask, default stream.
 *
 *   out  device, fp32, (B, NH, T, T) contiguous, fully overwritten.
 *   qkv  device, bf16, (B, T, 3, NH, HS) contiguous, HS = C / NH; read only.
 *   B, T, C, NH >= 1, C % NH == 0.
 *
 * Requirements (else CSA_ERR_ALIGN / CSA_ERR_UNSUPPORTED): qkv and out 16-byte
 * aligned; HS % 8 == 0 (the TMA row pitch of a head is HS*2 bytes and must be
 * a multiple of 16); HS <= 256. Any T >= 1 is accepted: rows and columns past
 * T are zero-filled on fetch and clipped on store. Scores are computed as
 * fp32 accumulations of exact bf16 products, then multiplied by the fp32
 * value of 1/sqrt(HS).
 */
csa_status trimul_forward(float* out, const void* qkv, int B, int T, int C, int NH);

/*
 * trimul_forward_ex -- as trimul_forward, with
 *   mask_bits  the 32-bit pattern written above the diagonal (CSA_MASK_NAN,
 *              CSA_MASK_NEG_INF or any other pattern);
 *   flags      CSA_TRIMUL_FULL or CSA_TRIMUL_LOWER_ONLY;
 *   stream     cudaStream_t (void*), NULL = default stream.
 */
csa_status trimul_forward_ex(float* out, const void* qkv, int B, int T, int C, int NH,
                             uint32_t mask_bits, uint32_t flags, void* stream);

/*
 * trimul_forward_f32 -- the causal score product over fp32 inputs, the
 * referee's own input type ("llm.c dev/cuda/trimat_forward.cu": trimul_cpu
 * takes const float* inp, and main fills it with fp32 random numbers), with no
 * rounding of the inputs to bf16.
 *
 *   out        device, fp32, (B, NH, T, T) contiguous; every element written
 *              (or only t2 <= t with CSA_TRIMUL_LOWER_ONLY).
 *   qkv        device, fp32, (B, T, 3, NH, HS) contiguous, HS = C / NH; read only.
 *   mask_bits, flags, stream   as trimul_forward_ex.
 *
 * Arithmetic: tcgen05 kind::tf32 with three products per input pair. Each
 * input x is split exactly into hi (x with its 13 lowest mantissa bits
 * cleared, a tf32 value: what the tensor core reads of x) and lo = x - hi;
 * each score accumulates
 * hi_q.hi_k + hi_q.lo_k + lo_q.hi_k in fp32, leaving out lo_q.lo_k, so each
 * product carries a relative error of a few units of 2^-20 on top of the fp32
 * accumulation, and the result is multiplied by the fp32 value of 1/sqrt(HS).
 *
 * Requirements (else CSA_ERR_ALIGN / CSA_ERR_UNSUPPORTED): qkv 16-byte and out
 * 4-byte aligned; HS % 4 == 0 (the TMA row pitch of a head is HS*4 bytes);
 * HS <= 256. Any T >= 1. Errors as trimul_forward_ex; nothing is written on
 * an argument error. The caller owns every buffer; nothing is allocated.
 */
csa_status trimul_forward_f32(float* out, const float* qkv, int B, int T, int C, int NH,
                              uint32_t mask_bits, uint32_t flags, void* stream);

/*
 * trimul_forward_noalloc -- trimul_forward_ex for callers that must not
 * allocate device memory. No passage of the pages has a counterpart: this
 * entry point exists for deployment, not for the method.
 *
 * Who needs it: code that runs where a new device allocation is not allowed or
 * not affordable -- under a memory manager that forbids allocations after
 * start-up, inside a region that must not trigger the device-wide
 * synchronisation cudaFree brings, or in plug-in hosts that only hand out
 * buffers. trimul_forward_ex itself never calls cudaMalloc either, but keeps
 * per-launch scheduling counters in a ring of slots; this variant instead
 * keeps its scratch -- the kernel's work-list counters (next position,
 * finished CTAs, next fill tile) -- in one fixed
 * 256-byte device array that every GPU loading the library holds until exit,
 * and calls no cudaMalloc, cudaFree or allocating library routine.
 *
 * Arguments, layouts, results and errors are those of trimul_forward_ex, plus:
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress); make that first call before any stream capture.
 *  - Every call clears the counters (cudaMemsetAsync on `stream`) before its
 *    kernel starts. All calls on a device share the array, so two calls whose
 *    kernels overlap on the GPU (different streams, no ordering) race and may
 *    leave output tiles unwritten; serialise them.
 *  - A problem whose tile list exceeds what the 32-bit counters can index
 *    (2^31 - 2^20 output tiles of 128 x 128) is rejected with CSA_ERR_SHAPE.
 */
csa_status trimul_forward_noalloc(float* out, const void* qkv, int B, int T, int C, int NH,
                                  uint32_t mask_bits, uint32_t flags, void* stream);

/*
 * dense_xwt -- Y = X W^T, default stream.
 *
 *   Y  device, fp32, [M, H] row-major, fully overwritten.
 *   X  device, bf16, [M, I] row-major; W device, bf16, [H, I] row-major.
 *   M, I, H >= 1, any values (no tile-multiple requirement).
 *
 * X and W need only 2-byte alignment. When I*2 is a multiple of 16 and both are
 * 16-byte aligned, tiles are fetched by TMA straight from X and W. Otherwise
 * (rows no tensor map can describe, e.g. I = 770) this call, which has no
 * workspace, fetches them with loader warps; dense_xwt_ws computes the same
 * layer faster with caller workspace. Y is written by TMA when H*4 is a
 * multiple of 16 and Y is 16-byte aligned (4-byte alignment required
 * otherwise). Tiles are 128 x BN (BN 64..256) per CTA, or, for problems large
 * enough (csa_dense_tiling), 256 x BN per cluster of two CTAs (tcgen05
 * cta_group::2) when the rows are fetched by TMA. Sums are fp32 accumulations of
 * exact bf16 products, in the same order on every fetch path and tiling (results
 * are bit-identical). Nothing is allocated.
 */
csa_status dense_xwt(float* Y, const void* X, const void* W, int M, int I, int H);

/* dense_xwt_ex -- as dense_xwt on `stream` (cudaStream_t as void*). */
csa_status dense_xwt_ex(float* Y, const void* X, const void* W, int M, int I, int H,
                        void* stream);

/*
 * dense_xwt_workspace_size -- bytes of device workspace dense_xwt_ws needs for
 * these operands, written to *bytes: 0 when tensor maps describe the rows of X
 * and W as they are (I*2 % 16 == 0, both 16-byte aligned), else
 * 256 + ceil256(M*P*2) + H*P*2 with P = I rounded up to a multiple of 64 (a
 * copy of X and W whose rows start on 128-byte boundaries, and alignment
 * slack). Depends on the pointers' alignment and the sizes only.
 * CSA_ERR_NULL / CSA_ERR_SHAPE as dense_xwt (then *bytes = 0).
 */
csa_status dense_xwt_workspace_size(const void* X, const void* W, int M, int I, int H,
                                    size_t* bytes);

/*
 * dense_xwt_ws -- dense_xwt with caller-owned scratch, on `stream`. Where no
 * tensor map can describe the rows of X and W, a first kernel copies them into
 * `workspace` as rows of pitch P (128-byte multiples) and the product kernel
 * fetches every tile from that copy by TMA, with zero fill past M, H and I --
 * the local padding of "DietCode tests/codegen/test_1_local_padding.py"
 * (bounds handled only where data is fetched and written back).
 *   workspace        device, 16-byte aligned, at least dense_xwt_workspace_size
 *                    bytes (else CSA_ERR_WORKSPACE / CSA_ERR_ALIGN, nothing
 *                    launched); may be NULL when that size is 0.
 *   workspace_bytes  its size.
 * The workspace needs no clearing, and its content after a call is unspecified.
 * It is in use until the call's kernels complete on `stream`: calls that may
 * overlap on the GPU need separate workspaces. Results are bit-identical to
 * dense_xwt on the same operands. Nothing is allocated.
 */
csa_status dense_xwt_ws(float* Y, const void* X, const void* W, int M, int I, int H,
                        void* workspace, size_t workspace_bytes, void* stream);

/*
 * dense_xwt_grouped -- Y[g] = X[g] W^T for g = 0 .. n-1, asynchronous on `stream`:
 * n dense layers that share W (device, bf16, [H, I]), I and H, computed by one
 * persistent launch over all their tiles (one launch per 48 problems), so that
 * a batch of dynamic-shape calls costs one launch instead of n.
 *   Y  host array of n device pointers: Y[g] fp32 [M[g], H] row-major, fully
 *      overwritten.
 *   X  host array of n device pointers: X[g] bf16 [M[g], I] row-major.
 *   M  host array of n row counts, each >= 1.
 * The host arrays are read during the call only. Results are bit-identical to n
 * dense_xwt calls. When I * 2 is not a multiple of 16, or W or some X[g] is not
 * 16-byte aligned, this call (no workspace) makes n dense_xwt launches instead;
 * dense_xwt_grouped_ws keeps such a batch in one grouped launch. Alignment: X[g]
 * and W 2-byte, Y[g] 4-byte (Y written by TMA when H * 4 % 16 == 0 and every Y[g]
 * is 16-byte aligned). CSA_ERR_NULL / CSA_ERR_SHAPE / CSA_ERR_ALIGN name the first
 * offending problem; nothing is launched then.
 */
csa_status dense_xwt_grouped(float* const* Y, const void* const* X, const void* W, const int* M,
                             int n, int I, int H, void* stream);

/*
 * dense_xwt_grouped_workspace_size -- bytes of device workspace
 * dense_xwt_grouped_ws needs for these operands, written to *bytes: 0 when
 * tensor maps describe the rows of W and of every X[g] as they are, else
 * 256 + ceil256(H*P*2) + sum_g ceil256(M[g]*P*2), P = I rounded up to 64.
 * CSA_ERR_NULL / CSA_ERR_SHAPE (then *bytes = 0).
 *
 * dense_xwt_grouped_ws -- dense_xwt_grouped with caller-owned scratch. Where no
 * tensor map can describe the rows (e.g. I = 770), one copy launch per 48
 * problems writes W's and the X[g]'s rows into `workspace` as 128-byte-aligned
 * rows (W once, then the problems in order), and the grouped launch reads them
 * from there, instead of one loader-warp dense_xwt per problem. Same bits as n
 * dense_xwt calls. workspace NULL is dense_xwt_grouped itself; otherwise it
 * must be 16-byte aligned and at least the size above (else CSA_ERR_ALIGN /
 * CSA_ERR_WORKSPACE, nothing launched). It is in use until the call's kernels
 * complete on `stream`. Nothing is allocated.
 */
csa_status dense_xwt_grouped_workspace_size(const void* const* X, const void* W, const int* M,
                                            int n, int I, int H, size_t* bytes);
csa_status dense_xwt_grouped_ws(float* const* Y, const void* const* X, const void* W,
                                const int* M, int n, int I, int H, void* workspace,
                                size_t workspace_bytes, void* stream);

/*
 * csa_set_dense_fetch -- process-wide fetch mode of dense_xwt_ws for rows that
 * no tensor map can describe (I*2 not a multiple of 16, or X / W not 16-byte
 * aligned):
 *   CSA_DENSE_FETCH_AUTO     copy the rows into the caller's workspace, then TMA;
 *   CSA_DENSE_FETCH_LOADERS  loader warps, as dense_xwt (the workspace unused).
 * Both modes give the same bits. Returns CSA_OK, or CSA_ERR_SHAPE for an
 * unknown mode (the mode is unchanged).
 */
#define CSA_DENSE_FETCH_AUTO    0
#define CSA_DENSE_FETCH_LOADERS 1
csa_status csa_set_dense_fetch(int mode);

/*
 * csa_dense_tiling -- the tiling dense_xwt / dense_xwt_ws choose for one problem of M
 * rows and H output columns whose rows are fetched by TMA (I * 2 % 16 == 0 and
 * 16-byte aligned operands, or rows realigned into a workspace), on a device or
 * stream with `sms` SMs: *bn = the tile width along H (64, 128, 192 or 256) and
 * *pairs = 1 when clusters of two CTAs compute 256-row tiles together (tcgen05
 * cta_group::2), else 0. Informational: a call falls back to single CTAs when no
 * cluster of two fits, and rows fetched by loader warps always use single CTAs.
 * Host only; returns CSA_OK, CSA_ERR_NULL or CSA_ERR_SHAPE.
 */
csa_status csa_dense_tiling(int M, int H, int sms, int* bn, int* pairs);

/*
 * csa_set_stream_sm_limit -- later calls of this library on `stream` (a
 * cudaStream_t; NULL is the legacy default stream) size their grids and tilings for
 * at most `max_sms` SMs: persistent kernels launch at most that many CTAs (CTA
 * pairs: max_sms / 2 clusters). Every kernel of this library holds a whole SM per
 * CTA (its shared memory), so a call limited to S SMs on one stream and a call
 * limited to the device's SM count minus S on another can run side by side on
 * disjoint SMs, as long as the first is launched first (clusters need whole pairs
 * of SMs). max_sms = 0 removes the limit; a limit above the device's SM count has
 * no effect. Results are the same bits under any limit. Limits are keyed by the
 * stream's handle value, process-wide, for at most 64 streams at once (then
 * CSA_ERR_BUSY); a stream destroyed with a limit set should have it removed
 * first, since a new stream may reuse the handle. Returns CSA_OK, CSA_ERR_SHAPE
 * for max_sms < 0, or CSA_ERR_BUSY.
 */
csa_status csa_set_stream_sm_limit(void* stream, int max_sms);

/* csa_get_stream_sm_limit -- the limit set on `stream` (0: none) into *max_sms. */
csa_status csa_get_stream_sm_limit(void* stream, int* max_sms);

/*
 * causal_softmax_forward -- the causal score rows of trimul_forward followed by
 * a softmax over t2 <= t, in one kernel (the scores never reach memory):
 *   att[b][h][t][t2] = exp(s[t2] - m) / sum_{u <= t} exp(s[u] - m)  for t2 <= t,
 *   att[b][h][t][t2] = 0                                               for t2 > t,
 * s = Q[b][h][t] . K[b][h][t2] / sqrt(HS), m = max_{u <= t} s[u]. The score is
 * the referee of "llm.c dev/cuda/trimat_forward.cu" (taken, as its comment
 * says, from the attention forward pass, where this softmax follows); the
 * softmax is the two-pass form of the "Smallem" article 5 (row maximum and sum
 * of exponentials, then normalisation).
 *   att  device, fp32, (B, NH, T, T) contiguous, fully overwritten.
 *   qkv  device, bf16, (B, T, 3, NH, HS), HS = C / NH, HS % 8 == 0, HS <= 128.
 * qkv 16-byte aligned, att 4-byte aligned. Asynchronous on `stream`.
 */
csa_status causal_softmax_forward(float* att, const void* qkv, int B, int T, int C, int NH,
                                  void* stream);

/*
 * batch_matmul_nt -- the unmasked, unscaled batched NT product of
 * "DietCode tests/codegen/test_1_local_padding.py" (test_local_padding_ii
 * docstring, BatchMatmulNT):
 *   Y[i][j][k] = sum_l X[i][j][l] * W[i][k][l]
 *   Y  device, fp32, [batch, T1, T2] row-major, fully overwritten.
 *   X  device, bf16, [batch, T1, D]; W device, bf16, [batch, T2, D].
 *   batch, T1, T2 >= 1 (any values: rows and columns past T1 / T2 are
 *   zero-filled on fetch and clipped on store), D % 8 == 0, D <= 256.
 * X and W 16-byte aligned, Y 4-byte aligned (TMA stores when T2 % 4 == 0 and Y
 * is 16-byte aligned). Same kernel as trimul_forward with every tile computed
 * and no mask or scale. Asynchronous on `stream` (cudaStream_t as void*).
 */
csa_status batch_matmul_nt(float* Y, const void* X, const void* W, int batch, int T1, int T2,
                           int D, void* stream);

/*
 * csa_get_status -- synchronises `stream`, then returns and clears the current
 * device's status word: CSA_OK, or CSA_ERR_TIMEOUT if a kernel's bounded wait
 * ran out since the last call. Returns CSA_ERR_CUDA if synchronisation fails.
 */
csa_status csa_get_status(void* stream);

/* csa_status_string -- static description of a status code (never NULL). */
const char* csa_status_string(csa_status s);

/* csa_last_error -- text of the last failure on this host thread ("" if none). */
const char* csa_last_error(void);

/* csa_version -- library version string, e.g. "0.1.0 sm_103a". */
const char* csa_version(void);

/*
 * Watchdog controls, for tests of the failure path (no GPU fault involved).
 *
 * csa_set_wait_limit_ns -- upper bound, in nanoseconds of %globaltimer, on
 *   every spin-wait inside the kernels (0 restores the default: 2e9 = 2 s, or
 *   the environment variable CSA_WAIT_LIMIT_NS when it holds a positive integer,
 *   read once at the first launch or query).
 * csa_get_wait_limit_ns -- the bound the next launch will use.
 * csa_debug_inject -- when nonzero, the next kernel launch (any entry point)
 *   withholds one hand-off in every CTA: the first operand load (score
 *   products, the softmax's first Q tile, the dense layer's TMA form) or the
 *   first stage arrival (the dense layer's loader-warp forms), so a bounded wait
 *   downstream runs out; the kernel records CSA_ERR_TIMEOUT and returns with its
 *   output incomplete. Consumed by that launch.
 */
void csa_set_wait_limit_ns(uint64_t ns);
uint64_t csa_get_wait_limit_ns(void);
void csa_debug_inject(int enable);

/*
 * Stream holds, for tests of launches that wait on the host (no GPU wait involved).
 *
 * csa_debug_hold_stream -- enqueues on `stream` a host function that returns once
 *   csa_debug_release_streams is called (or after 10 s): work enqueued behind it
 *   starts only then. CSA_ERR_CUDA if the host function cannot be enqueued.
 * csa_debug_release_streams -- releases every hold enqueued so far.
 */
csa_status csa_debug_hold_stream(void* stream);
void csa_debug_release_streams(void);

#ifdef __cplusplus
}
#endif

#endif /* CSA_GB300_H */
