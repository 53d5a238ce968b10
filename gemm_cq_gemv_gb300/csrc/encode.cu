// Offline / per-call quantizers: Lloyd-Max codebook fit (A1), CQ encode (A2),
// per-token int8 activations (A3) and Q4_0 quantize (A7).
//
// Each kernel follows the rounding order stated in cqgemv.h so that its output is
// bit-identical to the CPU oracle: explicit __dmul_rn / __dadd_rn / __ddiv_rn /
// __fdiv_rn / rintf, no fused multiply-add in any decision.

#include "common.cuh"

namespace cq {
namespace {

// ---------------------------------------------------------------------------------
// A1: Lloyd-Max Gaussian fit ("14MB 装下 45M 参数…", §一: Lloyd-Max on 400k Gaussian
// samples, 200 iterations).  One CTA of 1024 threads; the per-cell sums are reduced
// in a fixed order, so the result is deterministic.
// ---------------------------------------------------------------------------------
constexpr int kFitThreads = 1024;

__global__ void __launch_bounds__(kFitThreads)
lloyd_max_fit_kernel(const double* __restrict__ s, int64_t n, int L, int iters,
                     float* __restrict__ out) {
    __shared__ double lv[16];
    __shared__ double wsum[kFitThreads / 32][16];
    __shared__ unsigned long long wcnt[kFitThreads / 32][16];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid < L) lv[tid] = normcdfinv(((double)tid + 0.5) / (double)L);
    __syncthreads();
    for (int it = 0; it < iters; ++it) {
        double thr[15];
#pragma unroll
        for (int t = 0; t < 15; ++t) thr[t] = (t + 1 < L) ? (lv[t] + lv[t + 1]) / 2.0 : 0.0;
        double sum[16];
        unsigned long long cnt[16];
#pragma unroll
        for (int t = 0; t < 16; ++t) { sum[t] = 0.0; cnt[t] = 0ull; }
        for (int64_t i = tid; i < n; i += kFitThreads) {
            const double x = s[i];
            int c = 0;
#pragma unroll
            for (int t = 0; t < 15; ++t) c += (t + 1 < L && thr[t] < x) ? 1 : 0;
#pragma unroll
            for (int t = 0; t < 16; ++t) {
                if (c == t) { sum[t] = __dadd_rn(sum[t], x); cnt[t] += 1ull; }
            }
        }
        // warp butterfly (fixed order), then warps in index order
#pragma unroll
        for (int t = 0; t < 16; ++t) {
#pragma unroll
            for (int m = 16; m >= 1; m >>= 1) {
                sum[t] = __dadd_rn(sum[t], __shfl_xor_sync(0xffffffffu, sum[t], m));
                cnt[t] += __shfl_xor_sync(0xffffffffu, cnt[t], m);
            }
        }
        if (lane == 0) {
#pragma unroll
            for (int t = 0; t < 16; ++t) { wsum[warp][t] = sum[t]; wcnt[warp][t] = cnt[t]; }
        }
        __syncthreads();
        if (tid < L) {
            double ssum = 0.0;
            unsigned long long scnt = 0ull;
            for (int w = 0; w < kFitThreads / 32; ++w) {
                ssum = __dadd_rn(ssum, wsum[w][tid]);
                scnt += wcnt[w][tid];
            }
            if (scnt > 0ull) lv[tid] = __ddiv_rn(ssum, (double)scnt);
        }
        __syncthreads();
    }
    if (tid < L) out[tid] = __double2float_rn(lv[tid]);
}

// ---------------------------------------------------------------------------------
// A2: CQ encode.  One warp per 128-weight group; lane l holds positions 4l..4l+3.
// ---------------------------------------------------------------------------------
constexpr int kEncThreads = 256;

struct EncodeParams {
    const float* W;
    uint8_t* packed;
    uint16_t* norms;
    int64_t groups;   // N * K / 128
    int bits;         // bits of one packed index field
    int nlev;         // levels searched (2^bits, or 3 for the ternary code)
    float lv[16];
};

__global__ void __launch_bounds__(kEncThreads) cq_encode_kernel(const EncodeParams p) {
    __shared__ float wbuf[kEncThreads / 32][kGroup];
    __shared__ uint8_t ibuf[kEncThreads / 32][kGroup];
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int64_t warp = ((int64_t)blockIdx.x * kEncThreads + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * kEncThreads) >> 5;
    const int L = p.nlev;
    for (int64_t gi = warp; gi < p.groups; gi += nwarps) {
        const float4 w4 = *reinterpret_cast<const float4*>(p.W + gi * kGroup + 4 * lane);
        *reinterpret_cast<float4*>(&wbuf[wid][4 * lane]) = w4;
        double v0 = w4.x, v1 = w4.y, v2 = w4.z, v3 = w4.w;
        // natural-order butterflies: span 1 and 2 inside the lane ...
        double a0 = __dadd_rn(v0, v1), a1 = __dsub_rn(v0, v1);
        double a2 = __dadd_rn(v2, v3), a3 = __dsub_rn(v2, v3);
        v0 = __dadd_rn(a0, a2); v2 = __dsub_rn(a0, a2);
        v1 = __dadd_rn(a1, a3); v3 = __dsub_rn(a1, a3);
        // ... spans 4..64 across lanes (lower element a, upper b -> a + b, a - b)
#pragma unroll
        for (int m = 1; m <= 16; m <<= 1) {
            const bool upper = (lane & m) != 0;
            const double p0 = __shfl_xor_sync(0xffffffffu, v0, m);
            const double p1 = __shfl_xor_sync(0xffffffffu, v1, m);
            const double p2 = __shfl_xor_sync(0xffffffffu, v2, m);
            const double p3 = __shfl_xor_sync(0xffffffffu, v3, m);
            v0 = upper ? __dsub_rn(p0, v0) : __dadd_rn(v0, p0);
            v1 = upper ? __dsub_rn(p1, v1) : __dadd_rn(v1, p1);
            v2 = upper ? __dsub_rn(p2, v2) : __dadd_rn(v2, p2);
            v3 = upper ? __dsub_rn(p3, v3) : __dadd_rn(v3, p3);
        }
        __syncwarp();
        // ||w||^2 summed in index order by lane 0, then broadcast
        double nrm = 0.0;
        if (lane == 0) {
            double acc = 0.0;
            for (int i = 0; i < kGroup; ++i) {
                const double x = (double)wbuf[wid][i];
                acc = __dadd_rn(acc, __dmul_rn(x, x));
            }
            nrm = __dsqrt_rn(acc);
        }
        nrm = __shfl_sync(0xffffffffu, nrm, 0);
        int idx[4] = {0, 0, 0, 0};
        if (nrm > 0.0) {
            const double r[4] = {v0, v1, v2, v3};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const double v = __ddiv_rn(r[j], nrm);
                double best = fabs(__dsub_rn(v, (double)p.lv[0]));
                int bi = 0;
                for (int t = 1; t < L; ++t) {
                    const double d = fabs(__dsub_rn(v, (double)p.lv[t]));
                    if (d < best) { best = d; bi = t; }
                }
                idx[j] = bi;
            }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) ibuf[wid][4 * lane + j] = (uint8_t)idx[j];
        __syncwarp();
        // dense LSB-first bit stream: word w holds bits [32 w, 32 w + 32)
        const int nwords = 4 * p.bits;
        if (lane < nwords) {
            uint32_t word = 0u;
            const int lo = 32 * lane, hi = lo + 32;
            for (int i = lo / p.bits; i < kGroup; ++i) {
                const int pos = p.bits * i;
                if (pos >= hi) break;
                if (pos + p.bits <= lo) continue;
                const uint32_t val = ibuf[wid][i];
                const int off = pos - lo;
                word |= (off >= 0) ? (val << off) : (val >> (-off));
            }
            reinterpret_cast<uint32_t*>(p.packed + gi * (int64_t)(16 * p.bits))[lane] = word;
        }
        if (lane == 0) p.norms[gi] = f64_to_f16_bits_rne(nrm);
        __syncwarp();
    }
}

// ---------------------------------------------------------------------------------
// A3: per-token symmetric int8.  One CTA per token.
// ---------------------------------------------------------------------------------
constexpr int kA8Threads = 512;

__device__ __forceinline__ int8_t a8_code(float x, float s) {
    const float q = fminf(fmaxf(rintf(__fdiv_rn(x, s)), -127.0f), 127.0f);
    return (int8_t)(int)q;
}

// One CTA per token; 16-byte loads / 4-byte stores when the row allows it (K % 4 == 0).
__global__ void __launch_bounds__(kA8Threads)
a8_quantize_kernel(const float* __restrict__ X, int64_t K, int8_t* __restrict__ Xq,
                   float* __restrict__ scale) {
    __shared__ float red[kA8Threads / 32];
    pdl_trigger();
    pdl_wait();
    const int64_t t = blockIdx.x;
    const float* x = X + t * K;
    int8_t* xq = Xq + t * K;
    const bool vec = (K & 3) == 0;
    float amax = 0.0f;
    if (vec) {
        const float4* x4 = reinterpret_cast<const float4*>(x);
        for (int64_t k = threadIdx.x; k < K / 4; k += kA8Threads) {
            const float4 v = x4[k];
            amax = fmaxf(fmaxf(amax, fmaxf(fabsf(v.x), fabsf(v.y))), fmaxf(fabsf(v.z), fabsf(v.w)));
        }
    } else {
        for (int64_t k = threadIdx.x; k < K; k += kA8Threads) amax = fmaxf(amax, fabsf(x[k]));
    }
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, m));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
    __syncthreads();
    amax = 0.0f;
    for (int w = 0; w < kA8Threads / 32; ++w) amax = fmaxf(amax, red[w]);
    const float s = (amax > 0.0f) ? __fdiv_rn(amax, 127.0f) : 1.0f;
    if (vec) {
        const float4* x4 = reinterpret_cast<const float4*>(x);
        char4* q4 = reinterpret_cast<char4*>(xq);
        for (int64_t k = threadIdx.x; k < K / 4; k += kA8Threads) {
            const float4 v = x4[k];
            q4[k] = make_char4(a8_code(v.x, s), a8_code(v.y, s), a8_code(v.z, s), a8_code(v.w, s));
        }
    } else {
        for (int64_t k = threadIdx.x; k < K; k += kA8Threads) xq[k] = a8_code(x[k], s);
    }
    if (threadIdx.x == 0) scale[t] = s;
}

// ---------------------------------------------------------------------------------
// Grouped A8 for the attention side (Needle .cact page, §四: int8 KV cache, per-head A8
// quantization of the query, per-head A8 fake-quant of keys and values, one 4-byte scale
// per 32 cached values).  Every group of G consecutive features of a row gets the
// per-token rule of a8_quantize: s = float32(max |x|) / 127 (1 for an all-zero group),
// q = clip(rint(x / s), -127, 127); the fake-quant writes float32(q * s).  One warp per
// group, G / 32 values per lane.
// ---------------------------------------------------------------------------------
template <bool FAKE>
__global__ void __launch_bounds__(256)
a8_groups_kernel(const float* __restrict__ X, int64_t groups, int G, int8_t* __restrict__ codes,
                 float* __restrict__ scales, float* __restrict__ Y) {
    pdl_trigger();
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int64_t warp = ((int64_t)blockIdx.x * 256 + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * 256) >> 5;
    const int per = G >> 5;   // values per lane (G is a multiple of 32, at most 256)
    for (int64_t g = warp; g < groups; g += nwarps) {
        const float* x = X + g * G;
        float v[8];
        float am = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            v[i] = (i < per) ? x[i * 32 + lane] : 0.0f;
            am = fmaxf(am, fabsf(v[i]));
        }
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, m));
        const float s = (am > 0.0f) ? __fdiv_rn(am, 127.0f) : 1.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (i < per) {
                const int8_t q = a8_code(v[i], s);
                if constexpr (FAKE) Y[g * G + i * 32 + lane] = __fmul_rn((float)q, s);
                else codes[g * G + i * 32 + lane] = q;
            }
        }
        if constexpr (!FAKE) {
            if (lane == 0) scales[g] = s;
        }
    }
}

// ---------------------------------------------------------------------------------
// A7: Q4_0 quantize.  One thread per 32-weight block of a zero-padded row.
// ---------------------------------------------------------------------------------
__global__ void __launch_bounds__(256)
q4_0_quantize_kernel(const float* __restrict__ W, int64_t N, int64_t K, int64_t nblk,
                     uint8_t* __restrict__ out) {
    const int64_t bid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (bid >= N * nblk) return;
    const int64_t row = bid / nblk, blk = bid % nblk;
    const float* w = W + row * K + blk * 32;
    const int cnt = (K - blk * 32 < 32) ? (int)(K - blk * 32) : 32;
    float v[32];
    float amax = 0.0f;
#pragma unroll
    for (int k = 0; k < 32; ++k) {
        v[k] = (k < cnt) ? w[k] : 0.0f;
        amax = fmaxf(amax, fabsf(v[k]));
    }
    const float d = (amax > 0.0f) ? __fdiv_rn(amax, 8.0f) : 1.0f;
    // 18 bytes as nine little-endian 16-bit words (the block start is 2-byte aligned):
    // word 0 = fp16(d), word 1 + k = nibble bytes 2k and 2k+1.
    uint16_t* o = reinterpret_cast<uint16_t*>(out + bid * 18);
    o[0] = __half_as_ushort(__float2half_rn(d));
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        uint32_t word = 0u;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float q = fminf(fmaxf(rintf(__fdiv_rn(v[4 * k + j], d)), -8.0f), 7.0f);
            word |= (uint32_t)((int)q + 8) << (4 * j);
        }
        o[1 + k] = (uint16_t)word;
    }
}

inline int blocks_for(int64_t work, int per_block, int cap) {
    int64_t b = (work + per_block - 1) / per_block;
    if (b < 1) b = 1;
    return (int)(b > cap ? cap : b);
}

}  // namespace
}  // namespace cq

using namespace cq;

extern "C" cq_status cq_codebook_fit(const double* samples, int64_t n, int L, int iters,
                                     float* levels_out, void* stream) {
    if (!samples || !levels_out || n < 1 || L < 2 || L > 16 || iters < 0)
        return CQ_ERR_INVALID_ARG;
    lloyd_max_fit_kernel<<<1, kFitThreads, 0, as_stream(stream)>>>(samples, n, L, iters,
                                                                     levels_out);
    return check_launch();
}

extern "C" cq_status cq_encode(const float* W, int64_t N, int64_t K, int g, int b,
                               const cq_codebook* cbk, uint8_t* packed, uint16_t* norms,
                               void* stream) {
    if (!W || !cbk || !packed || !norms || N < 1 || K < 1) return CQ_ERR_INVALID_ARG;
    if (g != kGroup || K % kGroup != 0 || !cq_code_valid(b)) return CQ_ERR_INVALID_ARG;
    if (!aligned16(W) || !aligned16(packed) || !aligned16(norms)) return CQ_ERR_ALIGNMENT;
    EncodeParams p;
    p.W = W; p.packed = packed; p.norms = norms;
    p.groups = N * (K / kGroup);
    p.bits = cq_field_bits(b);
    p.nlev = cq_num_levels(b);
    cq_host_levels(p.lv, b, cbk);
    const int grid = blocks_for(p.groups, kEncThreads / 32, sm_count() * 64);
    cq_encode_kernel<<<grid, kEncThreads, 0, as_stream(stream)>>>(p);
    return check_launch();
}

extern "C" cq_status a8_quantize(const float* X, int64_t B, int64_t K, int8_t* Xq,
                                 float* scale, void* stream) {
    if (!X || !Xq || !scale || B < 1 || K < 1 || B > 2147483647LL) return CQ_ERR_INVALID_ARG;
    if (!aligned16(X) || !aligned16(Xq) || !aligned16(scale)) return CQ_ERR_ALIGNMENT;
    return launch_pdl(a8_quantize_kernel, dim3((unsigned)B), dim3(kA8Threads), 0, as_stream(stream), X, K, Xq,
                      scale);
}

extern "C" cq_status q4_0_quantize(const float* W, int64_t N, int64_t K, uint8_t* blocks,
                                   void* stream) {
    if (!W || !blocks || N < 1 || K < 1) return CQ_ERR_INVALID_ARG;
    if (!aligned16(W) || !aligned16(blocks)) return CQ_ERR_ALIGNMENT;
    const int64_t nblk = (K + 31) / 32;
    const int64_t total = N * nblk;
    const int64_t grid = (total + 255) / 256;
    if (grid > 2147483647LL) return CQ_ERR_UNSUPPORTED;
    q4_0_quantize_kernel<<<(unsigned)grid, 256, 0, as_stream(stream)>>>(W, N, K, nblk, blocks);
    return check_launch();
}

namespace {
cq_status a8_groups_args(const float* X, int64_t T, int64_t D, int G) {
    if (!X || T < 1 || D < 1 || G < 32 || G > 256 || G % 32 != 0 || D % G != 0) return CQ_ERR_INVALID_ARG;
    if (T > ((int64_t)1 << 40) / D) return CQ_ERR_UNSUPPORTED;
    return CQ_OK;
}
unsigned a8_groups_grid(int64_t groups) {
    int64_t grid = (groups + 7) / 8;
    const int64_t cap = (int64_t)sm_count() * 16;
    if (grid > cap) grid = cap;
    return (unsigned)(grid < 1 ? 1 : grid);
}
}  // namespace

extern "C" cq_status a8_quantize_groups(const float* X, int64_t T, int64_t D, int G, int8_t* codes,
                                        float* scales, void* stream) {
    cq_status st = a8_groups_args(X, T, D, G);
    if (st != CQ_OK) return st;
    if (!codes || !scales) return CQ_ERR_INVALID_ARG;
    if (!aligned16(X) || !aligned16(codes) || !aligned16(scales)) return CQ_ERR_ALIGNMENT;
    const int64_t groups = T * (D / G);
    return launch_pdl(a8_groups_kernel<false>, dim3(a8_groups_grid(groups)), dim3(256), 0, as_stream(stream), X,
                      groups, G, codes, scales, (float*)nullptr);
}

extern "C" cq_status a8_fake_quant_groups(const float* X, int64_t T, int64_t D, int G, float* Y,
                                          void* stream) {
    cq_status st = a8_groups_args(X, T, D, G);
    if (st != CQ_OK) return st;
    if (!Y) return CQ_ERR_INVALID_ARG;
    if (!aligned16(X) || !aligned16(Y)) return CQ_ERR_ALIGNMENT;
    const int64_t groups = T * (D / G);
    return launch_pdl(a8_groups_kernel<true>, dim3(a8_groups_grid(groups)), dim3(256), 0, as_stream(stream), X,
                      groups, G, (int8_t*)nullptr, (float*)nullptr, Y);
}
