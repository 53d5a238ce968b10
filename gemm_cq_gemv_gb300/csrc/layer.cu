// Fused decode chain: every matrix of one layer in one launch (CQ and Q4_0).
//
// A decoder layer stores its matrices one after another ("14MB 装下 45M 参数…", §三:
// weights pre-transposed to [out, in], layer-major) and decode multiplies each of them by
// an activation vector.  For a small model a launch per matrix costs more than the matrix
// (a 312 x 312 Q4_0 matrix is 55 KB, about 10 ns of HBM time), so these kernels take the
// whole list of a layer's problems - the ragged-N lm_head included, like the fast kernel
// the smolmaxxing page's kernel table runs it on - and run them in one launch whose grid
// follows the rows:
//
//   * work items are blocks of rows of one problem, numbered problem after problem; a
//     CTA takes a contiguous run of items, so it prepares the activations of a problem
//     once (usually) and reuses them for all its items of that problem;
//   * CQ: the CTA quantizes the float32 activations per token with the rule of
//     a8_quantize (s = fp32(amax) / 127, q = clip(rint(x / s), -127, 127), IEEE float32
//     divisions, bit for bit) and rotates them per 128-group (xr = Hu q, exact integers)
//     into shared memory; Q4_0: the CTA copies the float32 activations;
//   * a row is handled by G threads (G a power of two covering its 32-position chunks:
//     16 for K = 512 or K = 312, 32 above); thread j takes chunks j, j + G, ... and the G
//     partial sums are added by shuffles in a fixed order;
//   * codewords come from a 16-entry table with one copy per lane (conflict-free), the
//     activations from shared memory padded by one float per 32 (conflict-free when the
//     lanes of a warp read different chunks);
//   * products and sums are float32; the result is deterministic.
//
// Arithmetic per format:
//   CQ    y[t][o] = s_t / 128 * sum_j norm[o][j] * sum_i cb[idx[o][j][i]] * xr[t][128 j + i]
//   Q4_0  y[t][o] = sum_blocks fp32(d) * sum_k (nib - 8) * x[t][k]   (KMCU page, §2, §3;
//         nib - 8 is formed exactly, so an all-eight block adds exactly 0)

#include <mutex>

#include "common.cuh"

namespace cq {
namespace {

constexpr int kLThreads = 256;
constexpr int kLMaxProblems = CQ_LAYER_MAX_PROBLEMS;
constexpr int kLMaxK = CQ_LAYER_MAX_K;
constexpr int kLMaxTB = 2;
// activations of one token in shared memory: 32-position chunks, each padded to 33 floats
constexpr int kLChunkStride = 33;
constexpr size_t kLActFloats = (size_t)(kLMaxK / 32) * kLChunkStride;   // per token

struct LayerProblem {
    const uint8_t* w;        // CQ packed indices or Q4_0 blocks
    const uint16_t* norms;   // CQ group norms (unused for Q4_0)
    const float* X;          // [B][K]
    float* Y;                // [B][N]
    int64_t N;
    int K;
    int G;                   // threads per row (power of two, <= 32)
    int64_t item0;           // first work item of this problem
};

struct LayerParams {
    LayerProblem pr[kLMaxProblems];
    int count;
    int B;                   // tokens (1 or 2)
    int field;               // CQ: bits per index field
    int64_t items;           // total work items
    int64_t items_per_cta;
    float lv[16];            // CQ level table
};

__device__ __forceinline__ int find_problem(const LayerParams& p, int64_t item) {
    int q = 0;
    for (int i = 1; i < p.count; ++i)
        if (item >= p.pr[i].item0) q = i;
    return q;
}

// Sum over the G threads of a row (G a power of two, aligned groups within the warp).
__device__ __forceinline__ float group_sum(float v, int G) {
    for (int m = G >> 1; m >= 1; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
    return v;
}

// xr = Hu q for the groups of one token, by warps: lane l holds positions 4l..4l+3 of a
// 128-group (two butterfly stages in the lane, five across lanes); values are exact
// integers.  `a` holds q as floats (chunk-padded layout) and receives xr.
__device__ __forceinline__ void rotate_groups(float* a, int K, int warp, int nwarps, int lane) {
    const int G = K / kGroup;
    for (int g = warp; g < G; g += nwarps) {
        // position p of the group lives at chunk (p / 32), offset p % 32 (stride 33)
        auto at = [&](int pos) -> float& {
            const int gp = g * kGroup + pos;
            return a[(gp >> 5) * kLChunkStride + (gp & 31)];
        };
        float v0 = at(4 * lane), v1 = at(4 * lane + 1), v2 = at(4 * lane + 2), v3 = at(4 * lane + 3);
        float a0 = v0 + v1, a1 = v0 - v1, a2 = v2 + v3, a3 = v2 - v3;
        v0 = a0 + a2; v2 = a0 - a2; v1 = a1 + a3; v3 = a1 - a3;
#pragma unroll
        for (int m = 1; m <= 16; m <<= 1) {
            const bool upper = (lane & m) != 0;
            const float p0 = __shfl_xor_sync(0xffffffffu, v0, m);
            const float p1 = __shfl_xor_sync(0xffffffffu, v1, m);
            const float p2 = __shfl_xor_sync(0xffffffffu, v2, m);
            const float p3 = __shfl_xor_sync(0xffffffffu, v3, m);
            v0 = upper ? (p0 - v0) : (v0 + p0);
            v1 = upper ? (p1 - v1) : (v1 + p1);
            v2 = upper ? (p2 - v2) : (v2 + p2);
            v3 = upper ? (p3 - v3) : (v3 + p3);
        }
        __syncwarp();
        at(4 * lane) = v0; at(4 * lane + 1) = v1; at(4 * lane + 2) = v2; at(4 * lane + 3) = v3;
    }
}

// Block-wide maximum (non-negative values); `red` holds kLThreads / 32 floats.
__device__ __forceinline__ float block_max(float v, float* red) {
    for (int m = 16; m >= 1; m >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, m));
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    __syncthreads();   // red may still be read by the previous call
    if (lane == 0) red[w] = v;
    __syncthreads();
    float r = red[0];
    for (int i = 1; i < kLThreads / 32; ++i) r = fmaxf(r, red[i]);
    return r;
}

template <bool kCQ>
__global__ void __launch_bounds__(kLThreads) layer_gemv_kernel(const __grid_constant__ LayerParams p) {
    extern __shared__ __align__(16) float smem_l[];
    float* act = smem_l;                                   // [B][kLActFloats]
    float* tab = act + kLMaxTB * kLActFloats;              // [16][32] codewords, one copy per lane
    float* red = tab + 16 * 32;                            // [8] block reduction
    float* sc = red + kLThreads / 32;                      // [B] per-token scale s_t / 128
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    pdl_trigger();
    if (kCQ) {
        for (int i = tid; i < 16 * 32; i += kLThreads) {
            const int e = i >> 5;
            float v = 0.0f;
#pragma unroll
            for (int u = 0; u < 16; ++u) v = (u == e) ? p.lv[u] : v;
            tab[i] = v;
        }
    }
    // The weights are read before the wait for the previous kernel of the stream (they
    // come from kernels that release their dependents only at completion): the first
    // item's first chunk is requested, then the wait, then the activations.
    bool waited = false;
    const int64_t it0 = (int64_t)blockIdx.x * p.items_per_cta;
    int64_t it1 = it0 + p.items_per_cta;
    if (it1 > p.items) it1 = p.items;
    int cur = -1;
    for (int64_t it = it0; it < it1; ++it) {
        const int q = find_problem(p, it);
        const LayerProblem& pr = p.pr[q];
        const int K = pr.K;
        const int nch = (K + 31) / 32;                    // 32-position chunks (Q4_0 blocks)
        // this item's rows: rows_per_cta = kLThreads / G, one row per G threads; thread j of
        // a row takes chunks j, j + G, ...
        const int G = pr.G;
        const int rows = kLThreads / G;
        const int64_t row = (it - pr.item0) * rows + tid / G;
        const int j = tid & (G - 1);
        const bool live = row < pr.N && j < nch;
        // the first chunk's weights are requested before the activations are prepared, so
        // that the two memory round trips overlap
        const int f = kCQ ? p.field : 4;
        const int64_t rowbytes = kCQ ? (int64_t)(K / kGroup) * 16 * f : (int64_t)nch * 18;
        const uint8_t* wrow = pr.w + (live ? row : 0) * rowbytes;
        auto load_chunk = [&](int c, uint32_t (&wv)[5], uint32_t& sh, uint16_t& nb) {
            if (kCQ) {
                const uint32_t* src = reinterpret_cast<const uint32_t*>(wrow + (int64_t)c * 4 * f);
#pragma unroll
                for (int k = 0; k < 4; ++k) wv[k] = k < f ? __ldg(src + k) : 0u;
                wv[4] = 0u;
                sh = 0u;
                nb = __ldg(pr.norms + row * (K / kGroup) + (c >> 2));
            } else {
                // the 18-byte block (2-byte aligned) from the aligned words around it: at
                // offset 0 mod 4 its last two bytes are read as a half word, so that no
                // byte past the block is touched
                const uintptr_t a = reinterpret_cast<uintptr_t>(wrow + (int64_t)c * 18);
                const uint32_t* w4 = reinterpret_cast<const uint32_t*>(a & ~(uintptr_t)3);
                sh = (uint32_t)(a & 3) * 8u;   // 0 or 16
#pragma unroll
                for (int k = 0; k < 4; ++k) wv[k] = __ldg(w4 + k);
                wv[4] = sh ? __ldg(w4 + 4) : (uint32_t)__ldg(reinterpret_cast<const uint16_t*>(w4 + 4));
                nb = 0;
            }
        };
        uint32_t wv0[5] = {0u, 0u, 0u, 0u, 0u}, sh0 = 0u;
        uint16_t nb0 = 0;
        if (live) load_chunk(j, wv0, sh0, nb0);
        if (q != cur) {
            // prepare this problem's activations (the previous problem's are no longer read)
            if (!waited) {
                pdl_wait();
                waited = true;
            }
            __syncthreads();
            for (int t = 0; t < p.B; ++t) {
                const float* x = pr.X + (int64_t)t * K;
                float* a = act + (size_t)t * kLActFloats;
                for (int i = tid; i < nch * 32; i += kLThreads)
                    a[(i >> 5) * kLChunkStride + (i & 31)] = i < K ? x[i] : 0.0f;
                if (kCQ) {
                    float m = 0.0f;
                    for (int i = tid; i < K; i += kLThreads) m = fmaxf(m, fabsf(x[i]));
                    m = block_max(m, red);
                    const float s = m > 0.0f ? __fdiv_rn(m, 127.0f) : 1.0f;
                    for (int i = tid; i < K; i += kLThreads) {
                        float& v = a[(i >> 5) * kLChunkStride + (i & 31)];
                        v = fminf(fmaxf(rintf(__fdiv_rn(v, s)), -127.0f), 127.0f);
                    }
                    if (tid == 0) sc[t] = s * (1.0f / 128.0f);
                    __syncthreads();
                    rotate_groups(a, K, warp, kLThreads / 32, lane);
                }
            }
            __syncthreads();
            cur = q;
        }
        float accv[kLMaxTB] = {0.0f, 0.0f};
        if (live) {
            for (int c = j; c < nch; c += G) {
                uint32_t wv[5], sh;
                uint16_t nb;
                if (c == j) {
#pragma unroll
                    for (int k = 0; k < 5; ++k) wv[k] = wv0[k];
                    sh = sh0;
                    nb = nb0;
                } else {
                    load_chunk(c, wv, sh, nb);
                }
                float s0[kLMaxTB] = {0.0f, 0.0f}, s1[kLMaxTB] = {0.0f, 0.0f};
                if (kCQ) {
                    const float nrm = f16_bits_to_f32(nb);
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int pos = f * i;
                        uint32_t v = wv[pos >> 5] >> (pos & 31);
                        if ((pos & 31) + f > 32) v |= wv[(pos >> 5) + 1] << (32 - (pos & 31));
                        const float cw = tab[(v & ((1u << f) - 1u)) * 32 + lane];
#pragma unroll
                        for (int t = 0; t < kLMaxTB; ++t) {
                            if (t < p.B) {
                                const float xv = act[(size_t)t * kLActFloats + c * kLChunkStride + i];
                                if (i & 1) s1[t] = fmaf(cw, xv, s1[t]);
                                else s0[t] = fmaf(cw, xv, s0[t]);
                            }
                        }
                    }
#pragma unroll
                    for (int t = 0; t < kLMaxTB; ++t) accv[t] = fmaf(nrm, s0[t] + s1[t], accv[t]);
                } else {
                    const float d = f16_bits_to_f32((uint16_t)(wv[0] >> sh));
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const uint32_t nw = __funnelshift_rc(wv[k], wv[k + 1], sh + 16u);   // shift 16 or 32
#pragma unroll
                        for (int b = 0; b < 8; ++b) {
                            // nibble 8k + b: even index in the low half of byte b / 2;
                            // (2^23 + nib) - (2^23 + 8) = nib - 8, exactly
                            const float wq = __uint_as_float(0x4B000000u | ((nw >> (4 * b)) & 15u)) - 8388616.0f;
#pragma unroll
                            for (int t = 0; t < kLMaxTB; ++t) {
                                if (t < p.B) {
                                    const float xv = act[(size_t)t * kLActFloats + c * kLChunkStride + 8 * k + b];
                                    if (b & 1) s1[t] = fmaf(wq, xv, s1[t]);
                                    else s0[t] = fmaf(wq, xv, s0[t]);
                                }
                            }
                        }
                    }
#pragma unroll
                    for (int t = 0; t < kLMaxTB; ++t) accv[t] = fmaf(d, s0[t] + s1[t], accv[t]);
                }
            }
        }
#pragma unroll
        for (int t = 0; t < kLMaxTB; ++t) {
            const float v = group_sum(accv[t], G);
            if (t < p.B && j == 0 && row < pr.N)
                pr.Y[(int64_t)t * pr.N + row] = kCQ ? v * sc[t] : v;
        }
    }
}

size_t layer_smem_bytes() {
    return (kLMaxTB * kLActFloats + 16 * 32 + kLThreads / 32 + kLMaxTB) * sizeof(float);
}

int threads_per_row(int K) {
    const int nch = (K + 31) / 32;
    int G = 1;
    while (G < nch && G < 32) G <<= 1;
    return G;
}

template <bool kCQ>
cq_status run_layer(LayerParams& p, cudaStream_t st) {
    static bool attr[64] = {};
    static std::mutex mu;
    auto kern = layer_gemv_kernel<kCQ>;
    const size_t smem = layer_smem_bytes();
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return check_launch();
    if (dev < 0 || dev >= 64) return CQ_ERR_UNSUPPORTED;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!attr[dev]) {
            if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
                return check_launch();
            attr[dev] = true;
        }
    }
    // the grid follows the work: up to 3 CTAs per SM, each a contiguous run of items
    int64_t ctas = 3 * (int64_t)sm_count();
    if (ctas > p.items) ctas = p.items;
    p.items_per_cta = (p.items + ctas - 1) / ctas;
    const int64_t grid = (p.items + p.items_per_cta - 1) / p.items_per_cta;
    return launch_pdl(kern, dim3((unsigned)grid), dim3(kLThreads), smem, st, p);
}

// Fills the per-problem part of `p` (rows per item follow from G); false if a problem
// is out of range.
template <typename Prob, typename Get>
cq_status fill_problems(LayerParams& p, const Prob* probs, int count, int64_t B, Get get) {
    p.count = count;
    p.B = (int)B;
    int64_t items = 0;
    for (int i = 0; i < count; ++i) {
        LayerProblem& d = p.pr[i];
        const cq_status s = get(probs[i], d);
        if (s != CQ_OK) return s;
        d.G = threads_per_row(d.K);
        d.item0 = items;
        const int64_t rows = kLThreads / d.G;
        items += (d.N + rows - 1) / rows;
    }
    for (int i = count; i < kLMaxProblems; ++i) p.pr[i] = p.pr[0];
    p.items = items;
    return CQ_OK;
}

}  // namespace
}  // namespace cq

using namespace cq;

extern "C" cq_status cq_gemv_layer(const cq_gemv_problem* probs, int count, int g, int b,
                                   const cq_codebook* cbk, int64_t B, void* stream) {
    if (!probs || !cbk || count < 1 || B < 1) return CQ_ERR_INVALID_ARG;
    if (g != kGroup || !cq_code_valid(b)) return CQ_ERR_INVALID_ARG;
    if (count > kLMaxProblems || B > kLMaxTB) return CQ_ERR_UNSUPPORTED;
    LayerParams p;
    p.field = cq_field_bits(b);
    cq_host_levels(p.lv, b, cbk);
    const cq_status s = fill_problems(p, probs, count, B, [&](const cq_gemv_problem& q, LayerProblem& d) {
        if (!q.packed || !q.norms || !q.X || !q.Y || q.N < 1 || q.K < 1) return CQ_ERR_INVALID_ARG;
        if (q.K % kGroup != 0) return CQ_ERR_INVALID_ARG;
        if (q.K > kLMaxK || q.N > ((int64_t)1 << 40)) return CQ_ERR_UNSUPPORTED;
        if (!aligned16(q.packed) || !aligned16(q.norms) || !aligned16(q.X) || !aligned16(q.Y))
            return CQ_ERR_ALIGNMENT;
        d.w = q.packed; d.norms = q.norms; d.X = q.X; d.Y = q.Y; d.N = q.N; d.K = (int)q.K;
        return CQ_OK;
    });
    if (s != CQ_OK) return s;
    return run_layer<true>(p, as_stream(stream));
}

extern "C" cq_status q4_0_gemv_layer(const q4_0_gemv_problem* probs, int count, int64_t B, void* stream) {
    if (!probs || count < 1 || B < 1) return CQ_ERR_INVALID_ARG;
    if (count > kLMaxProblems || B > kLMaxTB) return CQ_ERR_UNSUPPORTED;
    LayerParams p;
    p.field = 4;
    for (int t = 0; t < 16; ++t) p.lv[t] = 0.0f;
    const cq_status s = fill_problems(p, probs, count, B, [&](const q4_0_gemv_problem& q, LayerProblem& d) {
        if (!q.blocks || !q.X || !q.Y || q.N < 1 || q.K < 1) return CQ_ERR_INVALID_ARG;
        if (q.K > kLMaxK || q.N > ((int64_t)1 << 40)) return CQ_ERR_UNSUPPORTED;
        if (!aligned16(q.blocks) || !aligned16(q.X) || !aligned16(q.Y)) return CQ_ERR_ALIGNMENT;
        d.w = q.blocks; d.norms = nullptr; d.X = q.X; d.Y = q.Y; d.N = q.N; d.K = (int)q.K;
        return CQ_OK;
    });
    if (s != CQ_OK) return s;
    return run_layer<false>(p, as_stream(stream));
}
