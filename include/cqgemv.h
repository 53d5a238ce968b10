/*
 * cqgemv.h - C ABI of the GB300 (sm_103a) low-bit GEMV / GEMM library (libcqgemv.so).
 *
 * Two weight formats:
 *
 *  CQ-WxA8 ("14MB 装下 45M 参数：拆解 Needle 的 .cact 单文件与 W4A8 量化魔法", §一 and §三;
 *  "免解析加载的秘诀：mmap 直读张量与 Needle 的秒级冷启动", section "mmap 之下张量按偏移直读"):
 *    a matmul weight W is stored pre-transposed [out = N, in = K]; each row is cut into
 *    groups of g = 128 along K; each group is rotated by the normalised Walsh-Hadamard
 *    transform, every rotated coordinate is replaced by the index of the nearest
 *    Lloyd-Max Gaussian codeword (b = 1..4 bits, or the ternary code b = 5), and the
 *    group's L2 norm is kept in FP16.  Reconstruction: w_group = (cb[idx] * norm / sqrt(g)) @ H, H = Hu / sqrt(g)
 *    (Hu the Sylvester Hadamard matrix, entries +-1).  Activations are int8 per token.
 *
 *  Q4_0 (Minueza-32M -> KMCU v1 page, §2 "Q4_0 量化" and §3 "行对齐到 32"):
 *    rows zero-padded to a multiple of 32; 32-weight blocks of 18 bytes: fp16 scale
 *    d = max_abs / 8 (little-endian, bytes 0..1), then 16 bytes of nibbles
 *    q + 8 with q = clip(rint(w / d), -8, 7), the low nibble holding the even index.
 *
 * Conventions shared by every call:
 *  - All array pointers are CUDA DEVICE memory owned by the caller; the library keeps no
 *    pointer after a call returns and allocates no device memory.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls only enqueue
 *    work: they are asynchronous and do not synchronise.
 *  - Kernels are launched with programmatic dependent launch: a kernel may start while
 *    the one before it on the stream finishes, and waits for it before it reads that
 *    kernel's outputs.  The batch-1 GEMVs start reading their packed weights before that
 *    wait, so weights must be complete when the kernel launched just before the GEMV
 *    starts: true for weights written by cq_encode or q4_0_quantize (neither releases
 *    its dependents early), by a copy, or by any kernel that does not trigger dependent
 *    launches itself.
 *  - Arguments are validated before anything is launched; a failed check returns an
 *    error status and launches nothing.
 *  - Row-major layouts; sizes are element counts unless named *_bytes.
 *  - Pointers must be 16-byte aligned (CQ_ERR_ALIGNMENT otherwise).
 *  - CQ_ERR_CUDA means a CUDA runtime call or launch failed; cq_last_cuda_error()
 *    returns its cudaError_t code.
 */
#ifndef CQGEMV_H
#define CQGEMV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define CQGEMV_ABI_VERSION 1
#define CQ_GROUP 128            /* CQ group size along K (Needle .cact page, §一) */
#define Q4_0_BLOCK 32           /* weights per Q4_0 block (KMCU page, §2)          */
#define Q4_0_BLOCK_BYTES 18     /* bytes per Q4_0 block  (KMCU page, §2)          */
/* The ternary CQ code (Needle mmap page, section "mmap 之下张量按偏移直读": bits = 5 selects
 * the fixed codebook {-c, 0, +c}).  The page gives no c; this library uses the
 * three-level Lloyd-Max level of N(0,1), c = 1.2240063619... (the root of
 * c = phi(c/2) / (1 - Phi(c/2))).  Indices 0, 1, 2 (-c, 0, +c) are stored in 2-bit fields
 * of the LSB-first stream, so a group takes 32 bytes, like b = 2; a field holding 3 never
 * comes out of cq_encode and reads as level 0. */
#define CQ_TERNARY 5

typedef enum cq_status {
    CQ_OK = 0,
    CQ_ERR_INVALID_ARG = 1,     /* bad shape, NULL pointer, g != 128, b not in 1..5, ... */
    CQ_ERR_ALIGNMENT = 2,       /* a pointer is not 16-byte aligned                      */
    CQ_ERR_UNSUPPORTED = 3,     /* no sm_103 device, or a size the kernels do not cover  */
    CQ_ERR_CUDA = 4,            /* CUDA runtime / launch error (see cq_last_cuda_error)  */
    CQ_ERR_DEVICE_TIMEOUT = 5,  /* a bounded device-side wait gave up                    */
    CQ_ERR_WORKSPACE = 6        /* workspace missing or smaller than *_workspace_bytes   */
} cq_status;

/* Codebook table: cb2[4] | cb3[8] | cb4[16], each ascending, in N(0,1) units - the
 * header table of the Needle .cact page, §一.  b = 1 ignores it and uses the analytic
 * +-sqrt(2/pi) of the Needle mmap page; b = CQ_TERNARY ignores it and uses {-c, 0, +c}.
 * Passed by pointer to HOST memory; copied by value into kernel parameters. */
typedef struct cq_codebook {
    float cb[28];
} cq_codebook;

/* Human-readable name of a status. Never NULL. */
const char* cq_status_string(cq_status s);
/* cudaError_t code of the last CQ_ERR_CUDA returned on the calling host thread (0 if none). */
int cq_last_cuda_error(void);
/* CQGEMV_ABI_VERSION of the loaded library. */
int cq_abi_version(void);

/* The level table the CQ kernels use for code b (Needle .cact page, §一: cb2 | cb3 | cb4
 * indexed by bit width; Needle mmap page: the fixed 1-bit and ternary codebooks), written
 * to levels_out [16] float32 in HOST memory: levels in index order, unused entries 0
 * (b = 1: -sqrt(2/pi), +sqrt(2/pi); b = CQ_TERNARY: -c, 0, +c, then 0 for the unused field
 * value 3; b = 2..4: the b-bit part of *cbk).  Host only: touches no device.
 * Errors: INVALID_ARG (b not in 1..5, levels_out NULL, cbk NULL for b = 2..4). */
cq_status cq_levels(int b, const cq_codebook* cbk, float* levels_out);

/* ---- A1: Lloyd-Max Gaussian codebook fit (Needle .cact page, §一: Lloyd-Max on
 * 400k Gaussian samples, 200 iterations).  Levels start at the N(0,1) quantiles
 * (t + 0.5) / L; one iteration puts thresholds at the midpoints of adjacent levels
 * (a sample equal to a threshold joins the lower cell) and moves each level to the
 * float64 mean of its cell (an empty cell keeps its level).
 *   samples    [n] float64, device
 *   L          number of levels, 2..16
 *   levels_out [L] float32, device, ascending
 * Errors: INVALID_ARG (n < 1, L out of range, iters < 0, NULL).  One CTA; meant for
 * offline use. */
cq_status cq_codebook_fit(const double* samples, int64_t n, int L, int iters,
                          float* levels_out, void* stream);

/* ---- A2: CQ encode (Needle .cact page, §一).  For each row o and group j:
 *   r = Hu @ w (float64 butterflies, natural order), n = sqrt(sum_i w_i^2) (float64,
 *   summed in index order, no fused multiply-add), idx_i = argmin_t |r_i / n - cb[t]|
 *   (float64; ties -> lowest index; n == 0 -> all indices 0), norm = fp16(n) (one
 *   round-to-nearest-even step from float64).
 *   W       [N][K] float32 ([out, in])
 *   packed  [N][K/128][16*f] uint8 with f = b (f = 2 for b = CQ_TERNARY): index i of a
 *           group in bits [f*i, f*i+f) of the group's little-endian bytes (b = 4: low
 *           nibble = even column)
 *   norms   [N][K/128] uint16 (IEEE binary16 bits)
 * Bit-exact with the CPU oracle.  Errors: INVALID_ARG (K % 128, g != 128, b not in
 * 1..5, N or K < 1, NULL), ALIGNMENT. */
cq_status cq_encode(const float* W, int64_t N, int64_t K, int g, int b,
                    const cq_codebook* cbk, uint8_t* packed, uint16_t* norms, void* stream);

/* ---- A3: per-token symmetric int8 activations (Needle .cact page, §一: ACT_BITS 8).
 *   s_t = float32(max_k |X[t][k]|) / 127 (IEEE float32 division; 1 if the token is
 *   all zero), Xq[t][k] = clip(rint(X[t][k] / s_t), -127, 127).
 *   X [B][K] float32 -> Xq [B][K] int8, scale [B] float32.  Bit-exact with the oracle.
 * Errors: INVALID_ARG (B or K < 1, NULL), ALIGNMENT. */
cq_status a8_quantize(const float* X, int64_t B, int64_t K, int8_t* Xq, float* scale,
                      void* stream);

/* ---- Grouped A8 for the attention side (Needle .cact page, §四: int8 KV cache, per-head A8
 * quantization of the query, per-head A8 fake-quant of keys and values, one 4-byte scale
 * per KV_GROUP = 32 cached values).  Every group of G consecutive features of a row of
 * X [T][D] float32 gets a8_quantize's per-token rule:
 *   s = float32(max |x|) / 127 (IEEE float32 division; 1 for an all-zero group),
 *   q = clip(rint(x / s), -127, 127).
 * a8_quantize_groups writes the codes [T][D] int8 and the scales [T][D/G] float32 (the
 * cache layout); a8_fake_quant_groups writes Y [T][D] = float32(q * s).  G is a multiple of
 * 32 up to 256 dividing D (a head of 32..256 features, or a KV group of 32).  Bit-exact with
 * the oracle.  Pointers 16-byte aligned.
 * Errors: INVALID_ARG, ALIGNMENT, UNSUPPORTED (T * D above 2^40), CUDA. */
cq_status a8_quantize_groups(const float* X, int64_t T, int64_t D, int G, int8_t* codes,
                             float* scales, void* stream);
cq_status a8_fake_quant_groups(const float* X, int64_t T, int64_t D, int G, float* Y, void* stream);

/* ---- A4 + A5: decode GEMV (Needle .cact page, §三: each output row streams along
 * the reduction axis; §一: reconstruction formula).  Computes, in float32,
 *   Y[t][o] = s_t * sum_j (norm[o][j] / 128) * sum_i cb[idx[o][j][i]] * xr[t][128 j + i]
 * with xr = Hu @ Xq per group (the rotated int8 activations, exact integers), which
 * equals (W_hat @ (s * Xq)^T)^T in real arithmetic because Hu is symmetric.
 * Four execution paths, chosen from the arguments:
 *   - b = 4, B <= 2, N >= 16, K a multiple of 1024: the CUDA-core GEMV on 16-bit integer
 *     codewords, C = rint(cb * S) with S = floor(32767 / max |cb|) (at most 4.2e-5
 *     absolute rounding of a Lloyd-Max level): exact integer dot products per 32
 *     positions, scaled by the fp16 group norm and summed in fp32.  The rotation happens
 *     inside the kernel; `workspace` is not touched.
 *   - b = 1, 2 or CQ_TERNARY, B = 1, N >= 16 x the number of SMs: the table-lookup kernel
 *     of cq_gemv_lut (below); `workspace` is not touched.
 *   - otherwise at B <= 2, or N not a multiple of 16: the CUDA-core GEMV on fp32
 *     codewords, fp32 products and accumulation; at B <= 2 the rotation happens inside
 *     the kernel, otherwise once per call into `workspace`, shared by every row.
 *   - B >= 3, N a multiple of 16 (any code): the tensor-core pipeline of cq_gemm with
 *     32-token tiles (4- and 2-bit rows reach shared memory per 64-index stage, 1- and
 *     3-bit rows per 128-index slab).  The weights are decoded once for all tokens; the operands are fp16
 *     (4- and 2-bit rows: fp16(fp16(cb) * norm); 1- and 3-bit rows: fp16(cb * norm); and
 *     xr * s_t / 128 in `workspace`), the accumulation fp32 (alternate 64-index stages of
 *     a tile into two partial sums, added in a fixed order).  The
 *     relative error stays within 1e-3 of the exact product; activations must satisfy
 *     max |X[t][k]| <= 65504 (fp16 range), and so must every group's norm times its
 *     largest codeword magnitude.  When the row tiles are too few to occupy the
 *     GPU, K is split in two: Y is zeroed on `stream` and both halves add their fp32
 *     partials into it (two addends on zero: the same sum in either order).
 *   packed, norms  as written by cq_encode (b = 1..4, or CQ_TERNARY: its 2-bit fields
 *                  run the 2-bit kernels on the level table {-c, 0, +c, 0})
 *   Xq [B][K] int8, scale [B] float32 (as written by a8_quantize)
 *   Y  [B][N] float32
 *   workspace      device scratch of at least cq_gemv_workspace_bytes(B, K) bytes
 * K is limited to 32768, N to 2^31 - 1024 and B to 2^30; on the tensor-core path also
 * ceil(B / 32) * ceil(N / 128) to 2^23 (CQ_ERR_UNSUPPORTED above).  Deterministic:
 * the same inputs give bit-identical outputs.
 * Errors: INVALID_ARG, ALIGNMENT, WORKSPACE, UNSUPPORTED, CUDA. */
size_t cq_gemv_workspace_bytes(int64_t B, int64_t K);
cq_status cq_gemv(const uint8_t* packed, const uint16_t* norms, int64_t N, int64_t K,
                  int g, int b, const cq_codebook* cbk, const int8_t* Xq,
                  const float* scale, int64_t B, float* Y, void* workspace,
                  size_t workspace_bytes, void* stream);

/* ---- A4 + A5 by table lookup, for narrow codes (b = 1, 2 or CQ_TERNARY): the 1-bit
 * lookup-table kernel of the smolmaxxing page (kernel table, Four-Russians / T-MAC style:
 * a 16-entry table per 4 activations) carried over to this format.  The same Y as cq_gemv:
 *   Y[t][o] = s_t * sum_j (norm[o][j] / 128) * sum_i cb[idx[o][j][i]] * xr[t][128 j + i].
 * For each token, every CTA rotates the activations (xr = Hu @ Xq per group) into shared
 * memory and tabulates, for every 4-bit nibble of the packed stream (four 1-bit or two
 * 2-bit indices), the 16 possible partial sums cb * xr over the positions it covers; a row
 * then costs one lookup and one fp32 add per nibble.  K is processed in ranges of 512
 * packed bytes per row (one table per range); rows stream through tensor copies.  Sums in
 * fp32 in a fixed order (deterministic); the result is within 1e-3 of the exact product
 * like cq_gemv's.
 *   packed, norms  as written by cq_encode for b = 1, 2 or CQ_TERNARY
 *   Xq [B][K] int8, scale [B] float32, Y [B][N] float32; all 16-byte aligned
 * No workspace.  Each token is one launch that reads the weights once (meant for batches
 * of 1 or 2).  K is limited to 2^24, N to 2^31 - 64 (the tensor copies address rows with
 * 32-bit coordinates), B to 2^30.
 * Errors: INVALID_ARG (NULL, g != 128, K % 128, b not in 1..5), UNSUPPORTED (b = 3 or 4,
 * sizes above the limits), ALIGNMENT, CUDA. */
cq_status cq_gemv_lut(const uint8_t* packed, const uint16_t* norms, int64_t N, int64_t K, int g,
                      int b, const cq_codebook* cbk, const int8_t* Xq, const float* scale,
                      int64_t B, float* Y, void* stream);

/* ---- A4 + A6: prefill GEMM on the tensor cores (Needle .cact page, §三: prefill is a
 * GEMM over the same [out, in] rows; §一: reconstruction formula).  Computes
 *   Y[t][o] = bf16( sum_k fp16(xr[t][k] * s_t / 128) * fp16(fp16(cb[idx[o][k]]) * norm[o][k/128]) )
 * with xr = Hu @ Xq per group (rotated once per call into `workspace`, fp16), tcgen05
 * MMA with fp32 accumulation in tensor memory.  The fp16 operands bound the range: a
 * token whose largest |activation| exceeds 65504, or a group whose norm times its largest
 * codeword does, overflows (the products become infinite).  Only b = 4 is implemented
 * (CQ_ERR_UNSUPPORTED for b = 1..3 and CQ_TERNARY).  N must be a multiple of 16 (INVALID_ARG); N and K
 * are limited to 2^24 (INVALID_ARG above), M to 2^30 (INVALID_ARG), and
 * ceil(M / 192) * ceil(N / 128) output tiles to 2^23 (UNSUPPORTED above).
 *   Xq [M][K] int8, scale [M] float32 (a8_quantize), Y [M][N] bf16 (uint16 bits)
 *   workspace: >= cq_gemm_workspace_bytes(M, K) bytes, 256-byte aligned
 * A device-side wait that does not complete within 2 s sets a device error flag and
 * the kernel returns early; cq_device_error() reports it as CQ_ERR_DEVICE_TIMEOUT.
 * Errors: INVALID_ARG, ALIGNMENT, WORKSPACE, UNSUPPORTED, CUDA. */
size_t cq_gemm_workspace_bytes(int64_t M, int64_t K);
cq_status cq_gemm(const uint8_t* packed, const uint16_t* norms, int64_t N, int64_t K, int g,
                  int b, const cq_codebook* cbk, const int8_t* Xq, const float* scale,
                  int64_t M, uint16_t* Y, void* workspace, size_t workspace_bytes,
                  void* stream);

/* One matrix of a grouped prefill launch: all pointers device memory; problems that
 * share an activation pass the same Xq pointer (and the same K), which is rotated once. */
typedef struct cq_gemm_problem {
    const uint8_t* packed;
    const uint16_t* norms;
    int64_t N;
    int64_t K;
    const int8_t* Xq;
    const float* scale;
    uint16_t* Y;
} cq_gemm_problem;

/* ---- A6 grouped: every problem of `probs` (host array of `count`) with the same M in
 * one persistent launch per 120 problems and 8 distinct activations (e.g. the 120
 * matrices of a 20-layer model, layer-major; up to 1024 problems per call, UNSUPPORTED
 * above).  Same arithmetic, limits and errors as cq_gemm; the workspace holds one
 * rotated copy per distinct Xq: cq_gemm_grouped_workspace_bytes(probs, count, M). */
size_t cq_gemm_grouped_workspace_bytes(const cq_gemm_problem* probs, int count, int64_t M);
cq_status cq_gemm_grouped(const cq_gemm_problem* probs, int count, int64_t M, int g, int b,
                          const cq_codebook* cbk, void* workspace, size_t workspace_bytes,
                          void* stream);

/* Failure-detection probe: enqueues on `stream` one single-thread kernel per compute unit
 * (GEMM pipeline, GEMV) whose bounded wait - the same device function the product kernels
 * use - waits on a barrier phase that nothing completes.  Each wait gives up after about
 * `timeout_ns` (1 us .. 10 s; the deadline is checked every 256 polls, each of which may
 * sleep up to 1 ms), raises its unit's device error word and returns: no fault, no hang.
 * A following cq_device_error() then reports CQ_ERR_DEVICE_TIMEOUT, and the context stays
 * usable.  Errors: INVALID_ARG (timeout out of range), CUDA. */
cq_status cq_probe_bounded_wait(uint64_t timeout_ns, void* stream);

/* Reports (and clears) the device error flags raised by a bounded wait that timed out
 * (2 s) in a GEMM or GEMV launch on the current device: CQ_ERR_DEVICE_TIMEOUT if any
 * was raised, else CQ_OK.  Synchronises `stream`. */
cq_status cq_device_error(void* stream);

/* ---- cq_gemv without a workspace (no counterpart in the format's description: a library
 * convenience).  Same computation, arguments and errors as cq_gemv, minus the
 * workspace, for callers that may not allocate device memory - typically code running
 * inside a host framework that owns every device allocation (an inference-server
 * plugin, an engine with a fixed memory budget) and forbids cudaMalloc while it runs.
 * The rotated activations go to a fixed scratch array inside the library image:
 *  - CQ_GEMV_NOALLOC_MAX_ELEMS floats (4 MiB), held on every GPU that loads the
 *    library until the process exits; B * K above it returns CQ_ERR_WORKSPACE;
 *  - the first call on a device looks up the array's device address (with that device
 *    current) and caches it: make that first call before any stream capture;
 *  - all calls share the array; each call writes what it reads, so no clearing is
 *    needed, but calls that overlap on the GPU (concurrent streams) race on it;
 *  - allocates nothing (no cudaMalloc / cudaFree, no allocating library routine). */
#define CQ_GEMV_NOALLOC_MAX_ELEMS (1u << 20)
cq_status cq_gemv_noalloc(const uint8_t* packed, const uint16_t* norms, int64_t N, int64_t K,
                          int g, int b, const cq_codebook* cbk, const int8_t* Xq,
                          const float* scale, int64_t B, float* Y, void* stream);

/* ---- Fused decode chain of one layer (Needle .cact page, §三: a layer's matrices are stored
 * layer-major, pre-transposed to [out, in], and decode multiplies each by an activation
 * vector; smolmaxxing page, kernel table: the ragged-N lm_head runs on the same kernel).
 * One launch covers every problem of `probs` (host array of `count` problems, at most
 * CQ_LAYER_MAX_PROBLEMS), for B = 1 or 2 tokens:
 *   cq_gemv_layer: for each problem, the per-token int8 quantization of its float32
 *     activations (the rule of a8_quantize, bit for bit), the rotation xr = Hu @ q per
 *     128-group and the product of cq_gemv,
 *       Y[t][o] = s_t * sum_j (norm[o][j] / 128) * sum_i cb[idx[o][j][i]] * xr[t][128 j + i],
 *     for any code b (1..4 or CQ_TERNARY), fp32 codewords, products and accumulation;
 *   q4_0_gemv_layer: for each problem, the product of q4_0_gemv,
 *       Y[t][o] = sum_blocks fp32(d) * sum_k (nib - 8) * X[t][k], float32.
 * Meant for the decode of small layers, where a launch per matrix costs more than the
 * matrix: the grid follows the rows (up to three 256-thread CTAs per SM, each on a
 * contiguous run of 256 / G-row blocks, G = the power of two of threads per row covering
 * its 32-position chunks), each CTA prepares the activations of the problems it serves
 * in shared memory, and no workspace is used.  Every sum has a fixed order, so reruns
 * are bit-identical.  Problems are independent (their outputs must not overlap their
 * inputs).
 *   packed, norms / blocks: as written by cq_encode / q4_0_quantize; N >= 1; K >= 1 with
 *   K % 128 == 0 for CQ; K <= CQ_LAYER_MAX_K; X [B][K] float32; Y [B][N] float32; every
 *   pointer 16-byte aligned.
 * Errors: INVALID_ARG (NULL, count < 1, B < 1, g != 128, K % 128 for CQ, a bad code),
 * UNSUPPORTED (count, B or K above the limits, N above 2^40), ALIGNMENT, CUDA. */
#define CQ_LAYER_MAX_PROBLEMS 16
#define CQ_LAYER_MAX_K 8192
typedef struct cq_gemv_problem {
    const uint8_t* packed;
    const uint16_t* norms;
    int64_t N;
    int64_t K;
    const float* X;
    float* Y;
} cq_gemv_problem;
cq_status cq_gemv_layer(const cq_gemv_problem* probs, int count, int g, int b,
                        const cq_codebook* cbk, int64_t B, void* stream);
typedef struct q4_0_gemv_problem {
    const uint8_t* blocks;
    int64_t N;
    int64_t K;
    const float* X;
    float* Y;
} q4_0_gemv_problem;
cq_status q4_0_gemv_layer(const q4_0_gemv_problem* probs, int count, int64_t B, void* stream);

/* ---- A7: Q4_0 quantize (KMCU page, §2, §3).
 *   W [N][K] float32 -> blocks [N][ceil(K/32) * 18] uint8; per block: d = amax / 8
 *   (float32; 1 if amax == 0), q = clip(rint(w / d), -8, 7) with float32 division,
 *   nibble = q + 8, byte k = nib[2k] | nib[2k+1] << 4, scale stored as fp16(d) (RNE).
 *   Columns K..32*ceil(K/32)-1 are zero padding (nibble 8).  Bit-exact with the oracle.
 * Errors: INVALID_ARG, ALIGNMENT (W only). */
cq_status q4_0_quantize(const float* W, int64_t N, int64_t K, uint8_t* blocks, void* stream);

/* ---- A8: Q4_0 decode GEMV (KMCU page, §2, §3: fixed-length 32 inner loop over
 * row-aligned blocks).  Y[t][o] = sum_blocks fp32(d) * sum_k (nib - 8) * X[t][k],
 * float32 accumulation; padding columns are skipped.  The activations of each 32-block
 * are held as 24-bit fixed-point integers, rint(x * 2^e) with the block's largest |x| in
 * [2^21, 2^22) (an error of at most 2^-23 of that value), so every block sum is exact in
 * int32: a block whose weights are all 0 contributes exactly 0, and an all-zero row or
 * token gives exactly 0.  A non-finite activation makes the outputs of its token NaN.
 *   blocks [N][ceil(K/32) * 18] uint8, X [B][K] float32, Y [B][N] float32 (all 16-byte
 *   aligned); K is limited to 32768, N to 2^31 - 1024 and B to 2^30 (CQ_ERR_UNSUPPORTED
 *   above).
 * Errors: INVALID_ARG, ALIGNMENT, UNSUPPORTED, CUDA. */
cq_status q4_0_gemv(const uint8_t* blocks, int64_t N, int64_t K, const float* X, int64_t B,
                    float* Y, void* stream);

/* ---- Q4_0 GEMM on the tensor cores (KMCU page, §2, §3 for the block format; the same
 * product as q4_0_gemv for M tokens at once: prefill, or a decode batch).  Computes
 *   Y[t][o] = sum_k fp16((nib[o][k] - 8) * d[o][k/32]) * fp16(X[t][k]),
 * with the products summed in float32 (tcgen05 MMA, fp32 accumulation in tensor memory).
 * `X` is converted once per call into `workspace` as fp16 [M][32 ceil(K/32)], zero past K;
 * each weight block is then read and decoded once per tile of up to 192 tokens (32 when
 * M <= 32; with few row tiles such calls split K in two and add both fp32 partials into Y,
 * zeroed first on `stream`).  The relative error stays within 1e-3 of the exact product; X must satisfy
 * max |X[t][k]| <= 65504 and the scales max |d| <= 8188 (fp16 range).
 *   blocks [N][ceil(K/32) * 18] uint8 (as written by q4_0_quantize), X [M][K] float32,
 *   Y [M][N] float32; all 16-byte aligned.
 *   workspace: >= q4_0_gemm_workspace_bytes(M, K) bytes, 256-byte aligned.
 * ceil(K/32) must be a multiple of 8 (whole 256-column slabs; CQ_ERR_UNSUPPORTED
 * otherwise: use q4_0_gemv); N and K are limited to 2^24, M to 2^30.
 * A device-side wait that does not complete within 2 s sets a device error flag and
 * the kernel returns early; cq_device_error() reports it as CQ_ERR_DEVICE_TIMEOUT.
 * Deterministic: the same inputs give bit-identical outputs.
 * Errors: INVALID_ARG, ALIGNMENT, WORKSPACE, UNSUPPORTED, CUDA. */
size_t q4_0_gemm_workspace_bytes(int64_t M, int64_t K);
cq_status q4_0_gemm(const uint8_t* blocks, int64_t N, int64_t K, const float* X, int64_t M,
                    float* Y, void* workspace, size_t workspace_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* CQGEMV_H */
