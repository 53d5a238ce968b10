// Table-lookup decode GEMV for narrow CQ codes (1-bit, 2-bit and the ternary code).
//
// The product is the one cq_gemv computes ("14MB 装下 45M 参数…", §一 and §三):
//   Y[t][o] = s_t / 128 * sum_j norm[o][j] * sum_i cb[idx[o][j][i]] * xr[t][128 j + i],
// xr = Hu @ Xq per 128-group.  Instead of looking up one codeword per index and
// multiplying it by an activation, the kernel precomputes, for every 4-bit nibble of the
// packed stream (four 1-bit indices, or two 2-bit ones), the 16 possible partial dot
// products with the activations that nibble covers; a row then costs one table lookup
// and one add per nibble.  This is the activation-table idea the smolmaxxing page
// describes for 1-bit CPU kernels: the table depends only on the activations, so it is
// built once per CTA and shared by every row.
//
// Layout of the work:
//   * one CTA of 16 warps per SM owns a contiguous block of rows;
//   * K is processed in ranges of 256 packed words per row (8192 positions at 1 bit,
//     4096 at 2 bits); for each range the CTA rotates the activations of the range into
//     shared memory, builds the table (128 KB) and streams its rows;
//   * a warp reads a row in 512-byte pieces: lane l loads words 4l..4l+3 of the piece
//     with one 16-byte load, so every lane's four words belong to one 128-group (1 bit)
//     or half of one (2 bits) and are scaled by that group's norm;
//   * the table is laid out so that lane l only ever reads bank l:
//       entry (piece sc, word v of the lane, nibble j of the word, value nib, lane l)
//       sits at float index ((sc * 4 + v) * 8 + j) * 512 + nib * 32 + l,
//     which makes every lookup of a warp conflict-free whatever the data;
//   * per-row partial sums stay in shared memory across ranges (one writer per row) and
//     are scaled by s_t / 128 once at the end; the order of every sum is fixed, so
//     reruns are bit-identical.
// There are no asynchronous copies and no barrier waits other than __syncthreads().

#include "common.cuh"

#include <mutex>

namespace cq {
namespace {

constexpr int kLutThreads = 512;                 // 16 warps
constexpr int kLutWarps = kLutThreads / 32;
constexpr int kPieceWords = 128;                 // words of a row read by one warp load
constexpr int kRangePieces = 2;                  // pieces per range
constexpr int kRangeWords = kRangePieces * kPieceWords;
constexpr int kPieceFloats = 4 * 8 * 16 * 32;    // table floats of one piece (64 KB)
constexpr int kTabFloats = kRangePieces * kPieceFloats;
constexpr int kRowBlock = 2048;                  // rows whose partials are kept at once
constexpr int kRowsPerWarp = 4;                  // rows a warp streams together

template <int F>
struct LutPlan {
    static constexpr int P = 4 / F;                          // positions per nibble
    static constexpr int range_pos = kRangeWords * 32 / F;   // positions per range
    static constexpr int pad = 32 * P;                       // one float of padding per pad
    static constexpr int xs_floats = range_pos + range_pos / pad;
    static constexpr size_t smem = (size_t)(kTabFloats + xs_floats + kRowBlock) * sizeof(float);
};
static_assert(LutPlan<1>::smem <= 227 * 1024 && LutPlan<2>::smem <= 227 * 1024, "shared memory");

struct LutParams {
    const uint8_t* packed;   // [N][words * 4] bytes
    const uint16_t* norms;   // [N][K / 128] fp16 bits
    const int8_t* Xq;        // [B][K]
    const float* scale;      // [B]
    float* Y;                // [B][N]
    int64_t N;
    int64_t rows_per_cta;
    int K;
    int words;               // packed 32-bit words per row: K * F / 32
    int nranges;             // ceil(words / kRangeWords)
    int t;                   // token of this launch
    float lv[4];             // levels by field value
};

// xs index of range position lp: one float of padding every 32 * P positions, so the
// table builders (lanes 32 * P positions apart) read 32 different banks.
template <int F>
__device__ __forceinline__ int xs_at(int lp) {
    return lp + lp / LutPlan<F>::pad;
}

template <int F>
__global__ void __launch_bounds__(kLutThreads, 1) cq_gemv_lut_kernel(const __grid_constant__ LutParams p) {
    using Pl = LutPlan<F>;
    constexpr int P = Pl::P;
    constexpr uint32_t kMask = (1u << F) - 1u;
    extern __shared__ __align__(16) float lsm[];
    float* tab = lsm;
    float* xs = tab + kTabFloats;
    float* part = xs + Pl::xs_floats;
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;

    const int64_t r_begin = (int64_t)blockIdx.x * p.rows_per_cta;
    const int64_t r_end = r_begin + p.rows_per_cta < p.N ? r_begin + p.rows_per_cta : p.N;
    const int64_t rowbytes = (int64_t)p.words * 4;
    const int G = p.K / kGroup;
    const int8_t* xq = p.Xq + (int64_t)p.t * p.K;
    float lv[1 << F];
#pragma unroll
    for (int u = 0; u < (1 << F); ++u) lv[u] = p.lv[u];
    bool built = false;

    for (int64_t rb0 = r_begin; rb0 < r_end; rb0 += kRowBlock) {
        const int nrb = (int)(r_end - rb0 < kRowBlock ? r_end - rb0 : kRowBlock);
        for (int r = 0; r < p.nranges; ++r) {
            const int rw0 = r * kRangeWords;                                  // first word
            const int nw = p.words - rw0 < kRangeWords ? p.words - rw0 : kRangeWords;
            if (!(built && p.nranges == 1)) {
                __syncthreads();   // every warp is done with the previous table
                // (1) xr = Hu @ q for the range's groups, one warp per group: lane l holds
                // positions 4l..4l+3; spans 1 and 2 inside the lane, 4..64 across lanes.
                // The values are integers below 2^24, exact in fp32.
                const int rp0 = rw0 * 32 / F;
                const int ngr = nw * 32 / F / kGroup;
                for (int gi = w; gi < ngr; gi += kLutWarps) {
                    const char4 c = *reinterpret_cast<const char4*>(xq + rp0 + gi * kGroup + 4 * lane);
                    float v0 = c.x, v1 = c.y, v2 = c.z, v3 = c.w;
                    const float a0 = v0 + v1, a1 = v0 - v1, a2 = v2 + v3, a3 = v2 - v3;
                    v0 = a0 + a2; v2 = a0 - a2; v1 = a1 + a3; v3 = a1 - a3;
#pragma unroll
                    for (int m = 1; m <= 16; m <<= 1) {
                        const bool upper = (lane & m) != 0;
                        const float q0 = __shfl_xor_sync(0xffffffffu, v0, m);
                        const float q1 = __shfl_xor_sync(0xffffffffu, v1, m);
                        const float q2 = __shfl_xor_sync(0xffffffffu, v2, m);
                        const float q3 = __shfl_xor_sync(0xffffffffu, v3, m);
                        v0 = upper ? (q0 - v0) : (v0 + q0);
                        v1 = upper ? (q1 - v1) : (v1 + q1);
                        v2 = upper ? (q2 - v2) : (v2 + q2);
                        v3 = upper ? (q3 - v3) : (v3 + q3);
                    }
                    const int lp = gi * kGroup + 4 * lane;
                    xs[xs_at<F>(lp)] = v0;
                    xs[xs_at<F>(lp + 1)] = v1;
                    xs[xs_at<F>(lp + 2)] = v2;
                    xs[xs_at<F>(lp + 3)] = v3;
                }
                __syncthreads();
                // (2) the table: warp task (sc, v, j), lane l -> nibble j of word
                // sc * 128 + 4 l + v of the range, its 16 partial dot products
                //   T[nib] = sum_q cb[field q of nib] * xr[position of field q]
                // (fields LSB-first: index i of the row sits in bits [F i, F i + F)).
                const int ntask = (nw + kPieceWords - 1) / kPieceWords * 32;
                for (int task = w; task < ntask; task += kLutWarps) {
                    const int sc = task >> 5, v = (task >> 3) & 3, j = task & 7;
                    const int wl = sc * kPieceWords + 4 * lane + v;
                    float x[P];
#pragma unroll
                    for (int q = 0; q < P; ++q) x[q] = 0.0f;
                    if (wl < nw) {
                        const int lp0 = (wl * 8 + j) * P;
#pragma unroll
                        for (int q = 0; q < P; ++q) x[q] = xs[xs_at<F>(lp0 + q)];
                    }
                    float* dst = tab + ((sc * 4 + v) * 8 + j) * 512 + lane;
#pragma unroll
                    for (int nib = 0; nib < 16; ++nib) {
                        float s = lv[nib & kMask] * x[0];
#pragma unroll
                        for (int q = 1; q < P; ++q) s = fmaf(lv[(nib >> (F * q)) & kMask], x[q], s);
                        dst[nib * 32] = s;
                    }
                }
                __syncthreads();
                built = true;
            }
            // (3) the rows: warp w takes rows w, w + 16, ... of the block, four at a time
            for (int i0 = w; i0 < nrb; i0 += kRowsPerWarp * kLutWarps) {
                float acc[kRowsPerWarp];
#pragma unroll
                for (int k = 0; k < kRowsPerWarp; ++k) acc[k] = 0.0f;
#pragma unroll
                for (int sc = 0; sc < kRangePieces; ++sc) {
                    const int wl = sc * kPieceWords + 4 * lane;
                    // whole 4-word runs lie inside or outside the range; a lane outside it
                    // reads nothing (its table entries may not have been built)
                    if (wl >= nw) continue;
                    const int wg = rw0 + wl;               // word within the row
                    uint4 wd[kRowsPerWarp];
                    float nr[kRowsPerWarp];
#pragma unroll
                    for (int k = 0; k < kRowsPerWarp; ++k) {
                        const int i = i0 + k * kLutWarps;
                        wd[k] = make_uint4(0u, 0u, 0u, 0u);
                        nr[k] = 0.0f;
                        if (i < nrb) {
                            const int64_t row = rb0 + i;
                            wd[k] = __ldg(reinterpret_cast<const uint4*>(p.packed + row * rowbytes + (int64_t)wg * 4));
                            nr[k] = f16_bits_to_f32(__ldg(p.norms + row * G + wg / (4 * F)));
                        }
                    }
                    const float* tl = tab + sc * kPieceFloats + lane;
#pragma unroll
                    for (int k = 0; k < kRowsPerWarp; ++k) {
                        const uint32_t wv[4] = {wd[k].x, wd[k].y, wd[k].z, wd[k].w};
                        float s0 = 0.0f, s1 = 0.0f;
#pragma unroll
                        for (int v = 0; v < 4; ++v)
#pragma unroll
                            for (int j = 0; j < 8; j += 2) {
                                s0 += tl[(v * 8 + j) * 512 + (((wv[v] >> (4 * j)) & 15u) << 5)];
                                s1 += tl[(v * 8 + j + 1) * 512 + (((wv[v] >> (4 * j + 4)) & 15u) << 5)];
                            }
                        acc[k] = fmaf(nr[k], s0 + s1, acc[k]);
                    }
                }
#pragma unroll
                for (int k = 0; k < kRowsPerWarp; ++k) {
                    float v = acc[k];
#pragma unroll
                    for (int m = 16; m >= 1; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
                    const int i = i0 + k * kLutWarps;
                    if (lane == 0 && i < nrb) part[i] = (r == 0) ? v : part[i] + v;
                }
            }
        }
        __syncthreads();   // all partials of the block are final
        const float ys = p.scale[p.t] * (1.0f / 128.0f);
        for (int i = tid; i < nrb; i += kLutThreads) p.Y[(int64_t)p.t * p.N + rb0 + i] = part[i] * ys;
        __syncthreads();   // part is rewritten by the next block
    }
}

template <int F>
cq_status run_lut(LutParams p, int64_t B, cudaStream_t st) {
    static bool attr[64] = {};
    static std::mutex mu;
    auto kern = cq_gemv_lut_kernel<F>;
    const size_t smem = LutPlan<F>::smem;
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
    const int64_t sms = sm_count();
    int64_t rpc = (p.N + sms - 1) / sms;
    if (rpc < kLutWarps) rpc = kLutWarps;
    p.rows_per_cta = rpc;
    const int64_t grid = (p.N + rpc - 1) / rpc;
    for (int64_t t = 0; t < B; ++t) {
        p.t = (int)t;
        cq_gemv_lut_kernel<F><<<(unsigned)grid, kLutThreads, smem, st>>>(p);
        const cq_status s = check_launch();
        if (s != CQ_OK) return s;
    }
    return CQ_OK;
}

}  // namespace
}  // namespace cq

using namespace cq;

extern "C" cq_status cq_gemv_lut(const uint8_t* packed, const uint16_t* norms, int64_t N, int64_t K,
                                 int g, int b, const cq_codebook* cbk, const int8_t* Xq,
                                 const float* scale, int64_t B, float* Y, void* stream) {
    if (!packed || !norms || !cbk || !Xq || !scale || !Y || N < 1 || K < 1 || B < 1)
        return CQ_ERR_INVALID_ARG;
    if (g != kGroup || K % kGroup != 0 || !cq_code_valid(b)) return CQ_ERR_INVALID_ARG;
    if (b != 1 && b != 2 && b != CQ_TERNARY) return CQ_ERR_UNSUPPORTED;
    if (K > (1 << 24) || N > ((int64_t)1 << 40) || B > (1 << 30)) return CQ_ERR_UNSUPPORTED;
    if (!aligned16(packed) || !aligned16(norms) || !aligned16(Xq) || !aligned16(scale) || !aligned16(Y))
        return CQ_ERR_ALIGNMENT;
    LutParams p;
    p.packed = packed; p.norms = norms; p.Xq = Xq; p.scale = scale; p.Y = Y;
    p.N = N; p.K = (int)K;
    const int f = cq_field_bits(b);
    p.words = (int)(K * f / 32);
    p.nranges = (p.words + kRangeWords - 1) / kRangeWords;
    p.rows_per_cta = 0;
    p.t = 0;
    float lv[16];
    cq_host_levels(lv, b, cbk);
    for (int u = 0; u < 4; ++u) p.lv[u] = lv[u];
    cudaStream_t st = as_stream(stream);
    return f == 1 ? run_lut<1>(p, B, st) : run_lut<2>(p, B, st);
}
