// Decode GEMV kernels: activation rotation (A4), CQ GEMV (A5) and Q4_0 GEMV (A8).
//
// Layout of the work ("14MB 装下 45M 参数…", §三: every output row is contiguous along
// the reduction axis, the axis the quant groups run along):
//   * a warp owns a tile of kRows output rows and walks K in segments of 1024
//     positions; lane l always covers positions [32 l, 32 l + 32) of a segment, so its
//     slice of the (rotated) activations stays in registers for every row of the tile
//     while the packed weights stream through with one coalesced load per lane per row;
//   * per-row partial dots are reduced across the warp with a butterfly that halves the
//     number of live rows at each step (9 shuffles for 8 rows);
//   * warps are persistent (grid-stride over tiles) and the activations of the call
//     sit in shared memory, loaded once per CTA.

#include <mutex>

#include "common.cuh"

namespace cq {
namespace {

constexpr int kThreads = 256;   // 8 warps
constexpr int kRows = 8;        // output rows per warp tile
constexpr int kSeg = 1024;      // positions per segment (32 lanes x 32)

// ---------------------------------------------------------------------------------
// A4: xr = Hu @ q per 128-group (Needle .cact page, §一, with H = Hu / sqrt(128) and
// H = H^T).  One warp per (token, group); values are small integers, exact in fp32.
// ---------------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads)
rotate_act_kernel(const int8_t* __restrict__ Xq, int64_t groups, float* __restrict__ xr) {
    const int lane = threadIdx.x & 31;
    const int64_t warp = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * kThreads) >> 5;
    for (int64_t gi = warp; gi < groups; gi += nwarps) {
        const char4 c = *reinterpret_cast<const char4*>(Xq + gi * kGroup + 4 * lane);
        float v0 = c.x, v1 = c.y, v2 = c.z, v3 = c.w;
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
        *reinterpret_cast<float4*>(xr + gi * kGroup + 4 * lane) = make_float4(v0, v1, v2, v3);
    }
}

// Butterfly reduction of 8 per-lane row partials: afterwards every lane holds the full
// sum of row ((lane >> 2) & 7).
__device__ __forceinline__ float reduce_rows8(const float (&a)[kRows], int lane) {
    float b[4], c[2];
    const bool u4 = lane & 16, u3 = lane & 8, u2 = lane & 4;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float send = u4 ? a[k] : a[k + 4];
        const float keep = u4 ? a[k + 4] : a[k];
        b[k] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
    }
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const float send = u3 ? b[k] : b[k + 2];
        const float keep = u3 ? b[k + 2] : b[k];
        c[k] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
    }
    float v = (u2 ? c[1] : c[0]) + __shfl_xor_sync(0xffffffffu, u2 ? c[0] : c[1], 4);
    v += __shfl_xor_sync(0xffffffffu, v, 2);
    v += __shfl_xor_sync(0xffffffffu, v, 1);
    return v;
}

// ---------------------------------------------------------------------------------
// A5: CQ GEMV.  Y[t][o] = s_t / 128 * sum_j norm[o][j] * sum_i cb[idx] * xr[t][128 j + i]
// ---------------------------------------------------------------------------------
struct CqGemvParams {
    const uint8_t* packed;
    const uint16_t* norms;
    const float* xr;      // [B][K] rotated activations
    const float* scale;   // [B]
    float* Y;             // [B][N]
    int64_t N;
    int K;
    int nseg;             // ceil(K / 1024)
    int t0;               // first token of this pass
    int ntok;             // tokens in this pass (<= TB)
    float lv[16];
};

template <int BITS>
__device__ __forceinline__ uint32_t extract_idx(const uint32_t (&w)[BITS], int i) {
    const int pos = BITS * i;
    const int wi = pos >> 5, sh = pos & 31;
    uint32_t v = w[wi] >> sh;
    if (sh + BITS > 32) v |= w[wi + 1] << (32 - sh);
    return v & ((1u << BITS) - 1u);
}

template <int BITS>
__device__ __forceinline__ void load_packed(uint32_t (&w)[BITS], const uint8_t* p) {
    if constexpr (BITS == 4) {
        const uint4 v = __ldcs(reinterpret_cast<const uint4*>(p));
        w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
    } else if constexpr (BITS == 2) {
        const uint2 v = __ldcs(reinterpret_cast<const uint2*>(p));
        w[0] = v.x; w[1] = v.y;
    } else {
#pragma unroll
        for (int k = 0; k < BITS; ++k) w[k] = __ldcs(reinterpret_cast<const uint32_t*>(p) + k);
    }
}

template <int BITS, int TB>
__global__ void __launch_bounds__(kThreads) cq_gemv_kernel(const CqGemvParams p) {
    extern __shared__ __align__(16) float smem[];
    float* lut = smem;                      // [16][32]: entry t replicated once per bank
    float* xs = smem + 16 * 32;             // [TB][nseg * 1024], zero padded
    const int lane = threadIdx.x & 31;
    const int segK = p.nseg * kSeg;
    constexpr int L = 1 << BITS;
    for (int i = threadIdx.x; i < 16 * 32; i += kThreads) {
        const int t = (i >> 5) & (L - 1);
        float v = 0.0f;
#pragma unroll
        for (int u = 0; u < 16; ++u) v = (u == t) ? p.lv[u] : v;
        lut[i] = v;
    }
    for (int i = threadIdx.x; i < TB * segK; i += kThreads) {
        const int t = i / segK, k = i - t * segK;
        xs[i] = (t < p.ntok && k < p.K) ? p.xr[(int64_t)(p.t0 + t) * p.K + k] : 0.0f;
    }
    __syncthreads();

    const int G = p.K / kGroup;
    const int64_t rowbytes = (int64_t)G * 16 * BITS;
    const int64_t ntiles = (p.N + kRows - 1) / kRows;
    const int64_t warp = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * kThreads) >> 5;
    const float* mylut = lut + lane;

    for (int64_t tile = warp; tile < ntiles; tile += nwarps) {
        const int64_t row0 = tile * kRows;
        float acc[TB][kRows];
#pragma unroll
        for (int t = 0; t < TB; ++t)
#pragma unroll
            for (int r = 0; r < kRows; ++r) acc[t][r] = 0.0f;

        for (int seg = 0; seg < p.nseg; ++seg) {
            const int pos0 = seg * kSeg + lane * 32;
            const bool active = pos0 < p.K;
            uint32_t w[kRows][BITS];
            float nrm[kRows];
#pragma unroll
            for (int r = 0; r < kRows; ++r) {
                const int64_t row = row0 + r;
                if (active && row < p.N) {
                    load_packed<BITS>(w[r], p.packed + row * rowbytes +
                                                (int64_t)seg * (128 * BITS) + lane * (4 * BITS));
                    nrm[r] = f16_bits_to_f32(__ldg(p.norms + row * G + seg * 8 + (lane >> 2)));
                } else {
#pragma unroll
                    for (int k = 0; k < BITS; ++k) w[r][k] = 0u;
                    nrm[r] = 0.0f;
                }
            }
            float x[TB][32];
#pragma unroll
            for (int t = 0; t < TB; ++t)
#pragma unroll
                for (int i = 0; i < 32; i += 4) {
                    const float4 v = *reinterpret_cast<const float4*>(xs + t * segK + pos0 + i);
                    x[t][i] = v.x; x[t][i + 1] = v.y; x[t][i + 2] = v.z; x[t][i + 3] = v.w;
                }
#pragma unroll
            for (int r = 0; r < kRows; ++r) {
                float dot[TB];
#pragma unroll
                for (int t = 0; t < TB; ++t) dot[t] = 0.0f;
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const float cw = mylut[extract_idx<BITS>(w[r], i) << 5];
#pragma unroll
                    for (int t = 0; t < TB; ++t) dot[t] = fmaf(cw, x[t][i], dot[t]);
                }
#pragma unroll
                for (int t = 0; t < TB; ++t) acc[t][r] = fmaf(nrm[r], dot[t], acc[t][r]);
            }
        }
#pragma unroll
        for (int t = 0; t < TB; ++t) {
            const float v = reduce_rows8(acc[t], lane);
            const int64_t row = row0 + ((lane >> 2) & 7);
            if ((lane & 3) == 0 && t < p.ntok && row < p.N) {
                const int tok = p.t0 + t;
                p.Y[(int64_t)tok * p.N + row] = v * (p.scale[tok] * (1.0f / 128.0f));
            }
        }
    }
}

// ---------------------------------------------------------------------------------
// A8: Q4_0 GEMV.  Lane l of a segment owns block (32 seg + l) of every row; the 18-byte
// blocks of a row segment are staged through shared memory with 16-byte loads.
// ---------------------------------------------------------------------------------
struct Q40GemvParams {
    const uint8_t* blocks;
    const float* X;       // [B][K]
    float* Y;             // [B][N]
    int64_t N;
    int K;
    int nblk;             // ceil(K / 32)
    int nseg;             // ceil(nblk / 32)
    int64_t total_bytes;  // N * nblk * 18
    int t0, ntok, B;
};

constexpr int kStage = 608;  // >= 37 chunks of 16 B, per row, per warp

template <int TB>
__global__ void __launch_bounds__(kThreads) q4_0_gemv_kernel(const Q40GemvParams p) {
    extern __shared__ __align__(16) float smem[];
    const int segK = p.nseg * kSeg;
    float* xs = smem;                                                      // [TB][segK]
    uint8_t* stage = reinterpret_cast<uint8_t*>(smem + TB * segK);         // [8 warps][kRows][kStage]
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    for (int i = threadIdx.x; i < TB * segK; i += kThreads) {
        const int t = i / segK, k = i - t * segK;
        xs[i] = (t < p.ntok && k < p.K) ? p.X[(int64_t)(p.t0 + t) * p.K + k] : 0.0f;
    }
    __syncthreads();
    uint8_t* mystage = stage + wid * (kRows * kStage);
    const int64_t rowbytes = (int64_t)p.nblk * 18;
    const int64_t ntiles = (p.N + kRows - 1) / kRows;
    const int64_t warp = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * kThreads) >> 5;
    const uintptr_t base_addr = reinterpret_cast<uintptr_t>(p.blocks);
    const uintptr_t end_addr = base_addr + (uintptr_t)p.total_bytes;

    for (int64_t tile = warp; tile < ntiles; tile += nwarps) {
        const int64_t row0 = tile * kRows;
        float acc[TB][kRows];
#pragma unroll
        for (int t = 0; t < TB; ++t)
#pragma unroll
            for (int r = 0; r < kRows; ++r) acc[t][r] = 0.0f;

        for (int seg = 0; seg < p.nseg; ++seg) {
            const int nb = min(32, p.nblk - seg * 32);
            int offs[kRows];
            __syncwarp();
#pragma unroll
            for (int r = 0; r < kRows; ++r) {
                const int64_t row = row0 + r;
                offs[r] = 0;
                if (row >= p.N) continue;
                const uintptr_t a = base_addr + (uintptr_t)(row * rowbytes + (int64_t)seg * 576);
                const uintptr_t start = a & ~(uintptr_t)15;
                offs[r] = (int)(a - start);
                const int chunks = (int)((a + (uintptr_t)nb * 18 - start + 15) >> 4);
                for (int c = lane; c < chunks; c += 32) {
                    const uintptr_t q = start + (uintptr_t)c * 16;
                    uint4 v;
                    if (q + 16 <= end_addr) {
                        v = __ldcs(reinterpret_cast<const uint4*>(q));
                    } else {
                        uint8_t tmp[16];
#pragma unroll
                        for (int k = 0; k < 16; ++k)
                            tmp[k] = (q + k < end_addr) ? *reinterpret_cast<const uint8_t*>(q + k) : 0;
                        v = make_uint4(tmp[0] | tmp[1] << 8 | tmp[2] << 16 | (uint32_t)tmp[3] << 24,
                                       tmp[4] | tmp[5] << 8 | tmp[6] << 16 | (uint32_t)tmp[7] << 24,
                                       tmp[8] | tmp[9] << 8 | tmp[10] << 16 | (uint32_t)tmp[11] << 24,
                                       tmp[12] | tmp[13] << 8 | tmp[14] << 16 | (uint32_t)tmp[15] << 24);
                    }
                    *reinterpret_cast<uint4*>(mystage + r * kStage + c * 16) = v;
                }
            }
            __syncwarp();
            if (lane < nb) {
                const int pos0 = seg * kSeg + lane * 32;
                float x[TB][32];
#pragma unroll
                for (int t = 0; t < TB; ++t)
#pragma unroll
                    for (int i = 0; i < 32; i += 4) {
                        const float4 v = *reinterpret_cast<const float4*>(xs + t * segK + pos0 + i);
                        x[t][i] = v.x; x[t][i + 1] = v.y; x[t][i + 2] = v.z; x[t][i + 3] = v.w;
                    }
#pragma unroll
                for (int r = 0; r < kRows; ++r) {
                    if (row0 + r >= p.N) continue;
                    const uint8_t* blk = mystage + r * kStage + offs[r] + lane * 18;
                    const uint16_t* h = reinterpret_cast<const uint16_t*>(blk);
                    const float d = f16_bits_to_f32(h[0]);
                    float s[TB];
#pragma unroll
                    for (int t = 0; t < TB; ++t) s[t] = 0.0f;
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const uint32_t two = h[1 + k];   // bytes 2k, 2k+1 -> 4 nibbles
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const uint32_t nib = (two >> (4 * j)) & 15u;
                            // (nib - 8) exactly: 2^23 + nib as a float, minus 2^23 + 8
                            const float wv = __uint_as_float(0x4B000000u | nib) - 8388616.0f;
#pragma unroll
                            for (int t = 0; t < TB; ++t) s[t] = fmaf(wv, x[t][4 * k + j], s[t]);
                        }
                    }
#pragma unroll
                    for (int t = 0; t < TB; ++t) acc[t][r] = fmaf(d, s[t], acc[t][r]);
                }
            }
        }
#pragma unroll
        for (int t = 0; t < TB; ++t) {
            const float v = reduce_rows8(acc[t], lane);
            const int64_t row = row0 + ((lane >> 2) & 7);
            if ((lane & 3) == 0 && t < p.ntok && row < p.N)
                p.Y[(int64_t)(p.t0 + t) * p.N + row] = v;
        }
    }
}

// Persistent grid: as many CTAs as fit, capped by the number of warp tiles.
int grid_for(const void* kern, size_t smem, int64_t ntiles) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem) != cudaSuccess ||
        per_sm < 1)
        return -1;
    int64_t want = (ntiles + (kThreads / 32) - 1) / (kThreads / 32);
    int64_t grid = (int64_t)per_sm * sm_count();
    if (want < grid) grid = want;
    return (int)(grid < 1 ? 1 : grid);
}

constexpr size_t kMaxSmem = 227 * 1024;

template <int BITS, int TB>
cq_status run_cq_gemv(CqGemvParams p, cudaStream_t st) {
    static bool attr = false;
    auto kern = cq_gemv_kernel<BITS, TB>;
    const size_t smem = (size_t)(16 * 32 + TB * p.nseg * kSeg) * sizeof(float);
    if (smem > kMaxSmem) return CQ_ERR_UNSUPPORTED;
    if (!attr) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kMaxSmem) !=
            cudaSuccess)
            return check_launch();
        attr = true;
    }
    const int64_t ntiles = (p.N + kRows - 1) / kRows;
    const int grid = grid_for((const void*)kern, smem, ntiles);
    if (grid < 0) return check_launch() == CQ_OK ? CQ_ERR_UNSUPPORTED : CQ_ERR_CUDA;
    kern<<<grid, kThreads, smem, st>>>(p);
    return check_launch();
}

template <int TB>
cq_status run_q4_0_gemv(Q40GemvParams p, cudaStream_t st) {
    static bool attr = false;
    auto kern = q4_0_gemv_kernel<TB>;
    const size_t smem = (size_t)TB * p.nseg * kSeg * sizeof(float) + (size_t)8 * kRows * kStage;
    if (smem > kMaxSmem) return CQ_ERR_UNSUPPORTED;
    if (!attr) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kMaxSmem) !=
            cudaSuccess)
            return check_launch();
        attr = true;
    }
    const int64_t ntiles = (p.N + kRows - 1) / kRows;
    const int grid = grid_for((const void*)kern, smem, ntiles);
    if (grid < 0) return check_launch() == CQ_OK ? CQ_ERR_UNSUPPORTED : CQ_ERR_CUDA;
    kern<<<grid, kThreads, smem, st>>>(p);
    return check_launch();
}

}  // namespace
}  // namespace cq

using namespace cq;

extern "C" size_t cq_gemv_workspace_bytes(int64_t B, int64_t K) {
    if (B < 1 || K < 1) return 0;
    return (size_t)B * (size_t)K * sizeof(float);
}

extern "C" cq_status cq_gemv(const uint8_t* packed, const uint16_t* norms, int64_t N, int64_t K,
                             int g, int b, const cq_codebook* cbk, const int8_t* Xq,
                             const float* scale, int64_t B, float* Y, void* workspace,
                             size_t workspace_bytes, void* stream) {
    if (!packed || !norms || !cbk || !Xq || !scale || !Y || N < 1 || K < 1 || B < 1)
        return CQ_ERR_INVALID_ARG;
    if (g != kGroup || K % kGroup != 0 || b < 1 || b > 4) return CQ_ERR_INVALID_ARG;
    if (K > (1 << 24) || N > ((int64_t)1 << 40)) return CQ_ERR_UNSUPPORTED;
    if (!aligned16(packed) || !aligned16(norms) || !aligned16(Xq) || !aligned16(scale) ||
        !aligned16(Y))
        return CQ_ERR_ALIGNMENT;
    if (!workspace || workspace_bytes < cq_gemv_workspace_bytes(B, K)) return CQ_ERR_WORKSPACE;
    if (!aligned16(workspace)) return CQ_ERR_ALIGNMENT;
    cudaStream_t st = as_stream(stream);
    float* xr = reinterpret_cast<float*>(workspace);
    const int64_t groups = B * (K / kGroup);
    {
        int64_t grid = (groups + 7) / 8;
        const int64_t cap = (int64_t)sm_count() * 16;
        if (grid > cap) grid = cap;
        rotate_act_kernel<<<(unsigned)grid, kThreads, 0, st>>>(Xq, groups, xr);
        const cq_status s = check_launch();
        if (s != CQ_OK) return s;
    }
    CqGemvParams p;
    p.packed = packed; p.norms = norms; p.xr = xr; p.scale = scale; p.Y = Y;
    p.N = N; p.K = (int)K; p.nseg = (int)((K + kSeg - 1) / kSeg);
    for (int t = 0; t < 16; ++t) p.lv[t] = 0.0f;
    if (b == 1) {
        const float c = 0.797884560802865355879892119868763737f;  // sqrt(2/pi)
        p.lv[0] = -c; p.lv[1] = c;
    } else {
        const int off = (b == 2) ? 0 : (b == 3) ? 4 : 12;
        for (int t = 0; t < (1 << b); ++t) p.lv[t] = cbk->cb[off + t];
    }
    // tokens per pass: 2 when the activations of two tokens fit in shared memory
    const int tb = ((size_t)2 * p.nseg * kSeg * sizeof(float) + 2048 <= kMaxSmem && B > 1) ? 2 : 1;
    for (int64_t t0 = 0; t0 < B; t0 += tb) {
        p.t0 = (int)t0;
        p.ntok = (int)((B - t0) < tb ? (B - t0) : tb);
        cq_status s;
        if (tb == 2) {
            switch (b) {
                case 1: s = run_cq_gemv<1, 2>(p, st); break;
                case 2: s = run_cq_gemv<2, 2>(p, st); break;
                case 3: s = run_cq_gemv<3, 2>(p, st); break;
                default: s = run_cq_gemv<4, 2>(p, st); break;
            }
        } else {
            switch (b) {
                case 1: s = run_cq_gemv<1, 1>(p, st); break;
                case 2: s = run_cq_gemv<2, 1>(p, st); break;
                case 3: s = run_cq_gemv<3, 1>(p, st); break;
                default: s = run_cq_gemv<4, 1>(p, st); break;
            }
        }
        if (s != CQ_OK) return s;
    }
    return CQ_OK;
}

extern "C" cq_status q4_0_gemv(const uint8_t* blocks, int64_t N, int64_t K, const float* X,
                               int64_t B, float* Y, void* stream) {
    if (!blocks || !X || !Y || N < 1 || K < 1 || B < 1) return CQ_ERR_INVALID_ARG;
    if (K > (1 << 24) || N > ((int64_t)1 << 40)) return CQ_ERR_UNSUPPORTED;
    if (!aligned16(blocks) || !aligned16(X) || !aligned16(Y)) return CQ_ERR_ALIGNMENT;
    Q40GemvParams p;
    p.blocks = blocks; p.X = X; p.Y = Y; p.N = N; p.K = (int)K;
    p.nblk = (int)((K + 31) / 32);
    p.nseg = (p.nblk + 31) / 32;
    p.total_bytes = N * (int64_t)p.nblk * 18;
    p.B = (int)B;
    cudaStream_t st = as_stream(stream);
    const size_t stage = (size_t)8 * kRows * kStage;
    const int tb = ((size_t)2 * p.nseg * kSeg * sizeof(float) + stage <= kMaxSmem && B > 1) ? 2 : 1;
    for (int64_t t0 = 0; t0 < B; t0 += tb) {
        p.t0 = (int)t0;
        p.ntok = (int)((B - t0) < tb ? (B - t0) : tb);
        const cq_status s = (tb == 2) ? run_q4_0_gemv<2>(p, st) : run_q4_0_gemv<1>(p, st);
        if (s != CQ_OK) return s;
    }
    return CQ_OK;
}

// ---------------------------------------------------------------------------------
// cq_gemv_noalloc: the decode GEMV for callers that may not allocate device memory.
//
// Some callers cannot hand this library a workspace: code that runs inside a host
// framework which owns every device allocation (an inference-server plugin, an engine
// that reserves its whole memory budget at start-up) may not call cudaMalloc while it
// executes, because an allocation can stall the device and breaks the fixed budget.
// This entry point keeps the rotated activations in a fixed scratch array that is
// part of the library image instead.
//
//  * The scratch is a file-scope __device__ array of CQ_GEMV_NOALLOC_MAX_ELEMS floats
//    (4 MiB).  Every GPU on which the library is loaded holds it until the process
//    exits.  B * K larger than that is rejected with CQ_ERR_WORKSPACE.
//  * Host code cannot use the array's name as a device address, so the first call on
//    each device looks the address up (cudaGetSymbolAddress, with that device current)
//    and caches it; make that first call before any stream capture.
//  * Every call shares the one array and it keeps the previous call's contents.  Each
//    call overwrites the B * K entries it reads before reading them, so nothing needs
//    clearing; but two calls that run at the same time on the GPU (different streams,
//    overlapping) race on the array.  Serialise them (one stream, or events).
//  * Nothing here allocates: no cudaMalloc / cudaFree, no library routine that does.
// ---------------------------------------------------------------------------------
namespace {

static __device__ __align__(256) float g_noalloc_xr[CQ_GEMV_NOALLOC_MAX_ELEMS];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
float* g_noalloc_ptr[kMaxDevices] = {nullptr};

cq_status noalloc_scratch(float** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) { set_last_cuda_error((int)e); return CQ_ERR_CUDA; }
    if (dev < 0 || dev >= kMaxDevices) return CQ_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (g_noalloc_ptr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_xr);   // current device = dev
        if (e != cudaSuccess || p == nullptr) {
            set_last_cuda_error((int)e);
            return CQ_ERR_CUDA;
        }
        g_noalloc_ptr[dev] = static_cast<float*>(p);
    }
    *out = g_noalloc_ptr[dev];
    return CQ_OK;
}

}  // namespace

extern "C" cq_status cq_gemv_noalloc(const uint8_t* packed, const uint16_t* norms, int64_t N,
                                     int64_t K, int g, int b, const cq_codebook* cbk,
                                     const int8_t* Xq, const float* scale, int64_t B, float* Y,
                                     void* stream) {
    if (!packed || !norms || !cbk || !Xq || !scale || !Y || N < 1 || K < 1 || B < 1)
        return CQ_ERR_INVALID_ARG;
    if (g != kGroup || K % kGroup != 0 || b < 1 || b > 4) return CQ_ERR_INVALID_ARG;
    if (B > (int64_t)CQ_GEMV_NOALLOC_MAX_ELEMS || K > (int64_t)CQ_GEMV_NOALLOC_MAX_ELEMS ||
        B * K > (int64_t)CQ_GEMV_NOALLOC_MAX_ELEMS)
        return CQ_ERR_WORKSPACE;
    if (!aligned16(packed) || !aligned16(norms) || !aligned16(Xq) || !aligned16(scale) ||
        !aligned16(Y))
        return CQ_ERR_ALIGNMENT;
    float* scratch = nullptr;
    const cq_status s = noalloc_scratch(&scratch);
    if (s != CQ_OK) return s;
    return cq_gemv(packed, norms, N, K, g, b, cbk, Xq, scale, B, Y, scratch,
                   (size_t)CQ_GEMV_NOALLOC_MAX_ELEMS * sizeof(float), stream);
}
