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
//   * K is processed in ranges of 128 packed words per row (512 bytes: 4096 positions at
//     1 bit, 2048 at 2 bits); for each range the CTA rotates the activations of the range
//     into shared memory and builds the table (64 KB) of that range;
//   * lane l of a warp owns words 4 l .. 4 l + 3 of the range, so its positions belong
//     to one 128-group (1 bit) or half of one (2 bits) and take that group's norm;
//   * the lookup address is one byte permute: the table starts at a 64 KB boundary, a
//     word masked with 0x0F0F0F0F holds its even nibbles in its bytes and one masked
//     with 0xF0F0F0F0 its odd nibbles (times 16), and the permute drops byte k of the
//     masked word into bits 8..15 of (table base | lane << 2).  So the entry of
//       even nibble 2k of word v, value n, lane l sits at (v * 4 + k) * 4096 + n * 256 + l * 4,
//       odd nibble 2k + 1, value n, lane l at      n * 4096 + (v * 4 + k) * 256 + 128 + l * 4
//     from the base (the odd entries fill the upper halves of the even ones' 256-byte
//     strides); what depends on the nibble's place is a constant offset of the shared
//     load, and lane l only ever reads bank l (no conflicts);
//   * a warp owns whole rows, 8 at a time (a row group): row group j belongs to CTA
//     j mod G and, in turn, to the CTA's warps, so every CTA holds the same number of
//     groups (+-1);
//   * packed rows arrive through a per-warp ring of four slots of two rows x one range
//     (1 KB), each filled by one tensor copy issued by one lane; a warp starts the copies
//     of a range before the table of that range is built; the group norms of the next row
//     group are loaded while the current one is looked up;
//   * a row group's eight 32-lane sums take one transposing butterfly; with one range the
//     sums are written out at once, with several they stay in shared memory across the
//     ranges (one writer per row, blocks of 2048 rows of the CTA at a time) and are
//     scaled by s_t / 128 at the end; the order of every sum is fixed, so reruns are
//     bit-identical.
// Every ring wait is bounded (the GEMV unit's device error word on expiry).

#include "gemv_pipe.cuh"

#include <mutex>

namespace cq {
namespace {

using namespace pipe;

constexpr int kLutThreads = 512;                 // 16 warps
constexpr int kLutWarps = kLutThreads / 32;
constexpr int kRangeWords = 128;                 // packed words of a row per range (512 bytes)
constexpr int kLutUnitRows = 2;                  // rows per staged unit
constexpr int kLutRing = 4;                      // slots per warp ring (slot = unit & 3)
constexpr uint32_t kLutUnitBytes = kLutUnitRows * kRangeWords * 4;   // 1 KB
constexpr uint32_t kLutTable = 65536;
constexpr int kBlockGroups = 256;                // row groups whose partials are kept at once
constexpr size_t kLutSmem = 227 * 1024;
static_assert(kLutRing == 4, "slot and phase arithmetic assume 4 slots");
static_assert(kRows == 4 * kLutUnitRows, "a row group is four units");

template <int F>
struct LutPlan {
    static constexpr int P = 4 / F;                          // positions per nibble
    static constexpr int range_pos = kRangeWords * 32 / F;   // positions per range
    static constexpr int pad = 32 * P;                       // one float of padding per pad
    static constexpr int xs_floats = range_pos + range_pos / pad;
};

struct LutParams {
    CUtensorMap pmap;        // packed rows as [N][words] uint32, box 128 x kLutUnitRows
    const uint16_t* norms;   // [N][K / 128] fp16 bits
    const int8_t* Xq;        // [B][K]
    const float* scale;      // [B]
    float* Y;                // [B][N]
    unsigned int* err;       // device error word
    int64_t N;
    int64_t groups_base;     // a CTA takes groups_base row groups, one more if
    int groups_extra;        //   blockIdx.x < groups_extra
    int K;
    int words;               // packed 32-bit words per row: K * F / 32
    int nranges;             // ceil(words / kRangeWords)
    int t;                   // token of this launch
    uint32_t smem_bytes;     // dynamic shared memory of the launch
    float lv[4];             // levels by field value
};

// xs index of range position lp: one float of padding every 32 * P positions, so the
// table builders (lanes 32 * P positions apart) read 32 different banks.
template <int F>
__device__ __forceinline__ int xs_at(int lp) {
    return lp + lp / LutPlan<F>::pad;
}

// (table base | lane << 2) with byte 1 replaced by byte K of the masked word
template <int K>
__device__ __forceinline__ uint32_t nib_addr(uint32_t masked, uint32_t lb) {
    uint32_t a;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(a) : "r"(masked), "r"(lb), "n"(0x7604 | (K << 4)));
    return a;
}
template <uint32_t OFF>
__device__ __forceinline__ float lds_at(uint32_t addr) {
    float v;
    asm volatile("ld.shared.f32 %0, [%1+%2];" : "=f"(v) : "r"(addr), "n"(OFF));
    return v;
}
__device__ __forceinline__ void sts_f32(uint32_t addr, float v) {
    asm volatile("st.shared.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

// The 8 lookups of one packed word (its even nibbles into se, its odd ones into so).
template <int V>
__device__ __forceinline__ void lookup_word(uint32_t wv, uint32_t lb, float& se, float& so) {
    const uint32_t lo = wv & 0x0F0F0F0Fu, hi = wv & 0xF0F0F0F0u;
    se += lds_at<(V * 4 + 0) * 4096>(nib_addr<0>(lo, lb));
    so += lds_at<(V * 4 + 0) * 256 + 128>(nib_addr<0>(hi, lb));
    se += lds_at<(V * 4 + 1) * 4096>(nib_addr<1>(lo, lb));
    so += lds_at<(V * 4 + 1) * 256 + 128>(nib_addr<1>(hi, lb));
    se += lds_at<(V * 4 + 2) * 4096>(nib_addr<2>(lo, lb));
    so += lds_at<(V * 4 + 2) * 256 + 128>(nib_addr<2>(hi, lb));
    se += lds_at<(V * 4 + 3) * 4096>(nib_addr<3>(lo, lb));
    so += lds_at<(V * 4 + 3) * 256 + 128>(nib_addr<3>(hi, lb));
}

template <int F>
__global__ void __launch_bounds__(kLutThreads, 1) cq_gemv_lut_kernel(const __grid_constant__ LutParams p) {
    using Pl = LutPlan<F>;
    constexpr int P = Pl::P;
    constexpr uint32_t kMask = (1u << F) - 1u;
    extern __shared__ __align__(128) unsigned char lsm[];
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    pdl_trigger();

    // shared plan: the table at a 64 KB boundary, everything else first-fit below and above
    const uint32_t sbase = smem_u32(lsm), send = sbase + p.smem_bytes;
    const uint32_t tbase = (sbase + 65535u) & ~65535u;
    SmemCarve cv;
    cv.ok = tbase + kLutTable <= send;
    cv.a = sbase; cv.a_end = tbase; cv.b = tbase + kLutTable; cv.b_end = send;
    const uint32_t bar_at = cv.take(kLutWarps * kLutRing * 8, 8);
    uint32_t ring_at;
    {   // the 16 rings (equal sizes: first-fit fills the space below the table, then above)
        constexpr uint32_t kRingB = kLutRing * kLutUnitBytes;
        const uint32_t a0 = (cv.a + 127u) & ~127u, b0 = (cv.b + 127u) & ~127u;
        const uint32_t na = a0 < cv.a_end ? (cv.a_end - a0) / kRingB : 0u;
        const uint32_t nb = (uint32_t)kLutWarps > na ? (uint32_t)kLutWarps - na : 0u;
        ring_at = (uint32_t)w < na ? a0 + (uint32_t)w * kRingB : b0 + ((uint32_t)w - na) * kRingB;
        if (na > 0u) cv.a = a0 + (na < (uint32_t)kLutWarps ? na : (uint32_t)kLutWarps) * kRingB;
        if (nb > 0u) {
            cv.b = b0 + nb * kRingB;
            if (cv.b > cv.b_end) cv.ok = false;
        }
    }
    const uint32_t xs_sa = cv.take(Pl::xs_floats * 4, 16);
    const uint32_t part_sa = cv.take(kBlockGroups * kRows * 4, 16);
    if (!cv.ok) {   // the launch's shared memory cannot hold the plan (host sizing error)
        if (tid == 0) atomicOr(p.err, 4u);
        return;
    }
    auto gen = [&](uint32_t a) { return lsm + (a - sbase); };
    uint64_t* rfull = reinterpret_cast<uint64_t*>(gen(bar_at)) + w * kLutRing;
    uint8_t* ring = gen(ring_at);
    float* xs = reinterpret_cast<float*>(gen(xs_sa));
    float* part = reinterpret_cast<float*>(gen(part_sa));
    if (tid == 0) prefetch_tensormap(&p.pmap);
    if (lane < kLutRing) mbar_init(&rfull[lane], 1);
    if (lane == 0) asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    __syncwarp();
    const uint32_t lb = tbase | ((uint32_t)lane << 2);
    const int G = p.K / kGroup;
    const int8_t* xq = p.Xq + (int64_t)p.t * p.K;
    float lv[1 << F];
#pragma unroll
    for (int u = 0; u < (1 << F); ++u) lv[u] = p.lv[u];
    const int64_t ncta = p.groups_base + ((int)blockIdx.x < p.groups_extra ? 1 : 0);
    const int64_t gstride = (int64_t)kLutWarps * gridDim.x;   // this warp's next group, in groups
    int64_t u_glob = 0;   // units this warp has consumed (its ring's slot and phase)
    // unit u of a range starting at word rw0, for the warp's groups from global group g0
    auto issue_at = [&](int64_t g0, int rw0, int u) {
        if (lane == 0) {
            const int d = (int)((u_glob + u) & (kLutRing - 1));
            const int64_t row = (g0 + (int64_t)(u >> 2) * gstride) * kRows + (u & 3) * kLutUnitRows;
            mbar_arrive_tx(&rfull[d], kLutUnitBytes);
            tma_box(ring + d * kLutUnitBytes, &p.pmap, rw0, (int)row, &rfull[d]);
        }
    };
    auto warp_units = [&](int64_t mb) {   // this warp's units per range in the block at mb
        const int nbg = (int)(ncta - mb < kBlockGroups ? ncta - mb : kBlockGroups);
        const int ngw = nbg > w ? (nbg - w + kLutWarps - 1) / kLutWarps : 0;
        return ngw * (kRows / kLutUnitRows);
    };
    // The packed rows are read before the wait for the previous kernel of the stream
    // (weights come from kernels that release their dependents only at completion): the
    // first range's first copies go out here, the activations are read after the wait.
    {
        const int nu0 = ncta > 0 ? warp_units(0) : 0;
        for (int u = 0; u < kLutRing - 1 && u < nu0; ++u) issue_at(blockIdx.x + (int64_t)w * gridDim.x, 0, u);
    }
    pdl_wait();   // the activations may come from the previous kernel
    const float yscale = p.scale[p.t] * (1.0f / 128.0f);
    bool built = false;
    // this warp's int8 activations of a range (its groups w and w + 16), loaded one range
    // ahead so a table rebuild does not wait for them
    constexpr int kGpw = LutPlan<F>::range_pos / kGroup / kLutWarps;   // groups per warp (2 or 1)
    char4 xpre[kGpw];
    auto load_acts = [&](int r) {
        const int rw = r * kRangeWords;
        const int n = p.words - rw < kRangeWords ? p.words - rw : kRangeWords;
        const int ngr = n * 32 / F / kGroup;
#pragma unroll
        for (int j = 0; j < kGpw; ++j) {
            const int gi = w + j * kLutWarps;
            xpre[j] = gi < ngr ? *reinterpret_cast<const char4*>(xq + rw * 32 / F + gi * kGroup + 4 * lane)
                               : make_char4(0, 0, 0, 0);
        }
    };
    load_acts(0);
    for (int64_t mb = 0; mb < ncta; mb += kBlockGroups) {
        const int nbg = (int)(ncta - mb < kBlockGroups ? ncta - mb : kBlockGroups);
        const int ngw = nbg > w ? (nbg - w + kLutWarps - 1) / kLutWarps : 0;   // this warp's groups
        // group i of this warp in the block is the CTA's group m = mb + w + 16 i, global
        // group g0 + i * gstride (rows from 8 times that)
        const int64_t g0 = blockIdx.x + (mb + w) * (int64_t)gridDim.x;
        for (int r = 0; r < p.nranges; ++r) {
            const int rw0 = r * kRangeWords;
            const int nw = p.words - rw0 < kRangeWords ? p.words - rw0 : kRangeWords;
            const int nunits = ngw * (kRows / kLutUnitRows);
            auto issue = [&](int u) { issue_at(g0, rw0, u); };
            // the first copies of the range go out before its table is built (those of the
            // first range of the first block before the dependent-launch wait)
            if (mb > 0 || r > 0) {
                __syncwarp();
                if (lane == 0) fence_proxy_async();   // earlier reads of the slots are done
                for (int u = 0; u < kLutRing - 1 && u < nunits; ++u) issue(u);
            }
            if (!(built && p.nranges == 1)) {
                __syncthreads();   // every warp is done with the previous table
                // (1) xr = Hu @ q for the range's groups, one warp per group: lane l holds
                // positions 4l..4l+3; spans 1 and 2 inside the lane, 4..64 across lanes.
                // The values are integers below 2^24, exact in fp32.
                const int ngr = nw * 32 / F / kGroup;
#pragma unroll
                for (int j = 0; j < kGpw; ++j) {
                    const int gi = w + j * kLutWarps;
                    if (gi >= ngr) continue;
                    const char4 c = xpre[j];
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
                // (2) the table: warp task (v, j), lane l -> nibble j of word 4 l + v of
                // the range, its 16 partial dot products
                //   T[nib] = sum_q cb[field q of nib] * xr[position of field q]
                // (fields LSB-first: index i of the row sits in bits [F i, F i + F)); words
                // past the range get zeros (the tensor copies read them as zero words)
                for (int task = w; task < 32; task += kLutWarps) {
                    const int v = task >> 3, j = task & 7;
                    const int wl = 4 * lane + v;
                    float x[P];
#pragma unroll
                    for (int q = 0; q < P; ++q) x[q] = 0.0f;
                    if (wl < nw) {
                        const int lp0 = (wl * 8 + j) * P;
#pragma unroll
                        for (int q = 0; q < P; ++q) x[q] = xs[xs_at<F>(lp0 + q)];
                    }
                    const uint32_t k4 = (uint32_t)(v * 4 + (j >> 1));
                    const uint32_t dst = (j & 1) ? tbase + k4 * 256u + 128u + (uint32_t)lane * 4u
                                                 : tbase + k4 * 4096u + (uint32_t)lane * 4u;
                    const uint32_t step = (j & 1) ? 4096u : 256u;
#pragma unroll
                    for (int nib = 0; nib < 16; ++nib) {
                        float s = lv[nib & kMask] * x[0];
#pragma unroll
                        for (int q = 1; q < P; ++q) s = fmaf(lv[(nib >> (F * q)) & kMask], x[q], s);
                        sts_f32(dst + (uint32_t)nib * step, s);
                    }
                }
                __syncthreads();
                built = true;
                if (p.nranges > 1) load_acts(r + 1 < p.nranges ? r + 1 : 0);   // the next rebuild's
            }
            // (3) the rows: units of two rows, the next three in flight; the norms of the
            // next row group loaded while the current one is looked up
            const bool lane_in = 4 * lane < nw;
            const int gcol = (rw0 + 4 * lane) * 32 / F / kGroup;   // this lane's 128-group
            // (the raw fp16 bits are kept until the group starts, so the loads do not stall)
            auto load_norms = [&](int i, uint32_t (&nr)[kRows]) {
                const int64_t row0 = (g0 + (int64_t)i * gstride) * kRows;
#pragma unroll
                for (int k = 0; k < kRows; ++k) {
                    nr[k] = 0u;
                    if (i < ngw && lane_in && row0 + k < p.N) nr[k] = __ldg(p.norms + (row0 + k) * G + gcol);
                }
            };
            float ncur[kRows], acc[kRows];
            uint32_t nnext[kRows];
            load_norms(0, nnext);
            for (int i = 0; i < ngw; ++i) {
#pragma unroll
                for (int k = 0; k < kRows; ++k) ncur[k] = f16_bits_to_f32((uint16_t)nnext[k]);
                load_norms(i + 1, nnext);
#pragma unroll
                for (int h = 0; h < kRows / kLutUnitRows; ++h) {
                    const int u = 4 * i + h;
                    if (u + kLutRing - 1 < nunits) {
                        __syncwarp();   // every lane is done with the slot about to be refilled
                        if (lane == 0) fence_proxy_async();
                        issue(u + kLutRing - 1);
                    }
                    const int d = (int)((u_glob + u) & (kLutRing - 1));
                    mbar_wait(&rfull[d], (uint32_t)((u_glob + u) >> 2) & 1u, p.err);
                    const uint8_t* sp = ring + d * kLutUnitBytes + lane * 16;
#pragma unroll
                    for (int rr = 0; rr < kLutUnitRows; ++rr) {
                        const uint4 wq = *reinterpret_cast<const uint4*>(sp + rr * (kRangeWords * 4));
                        float se = 0.0f, so = 0.0f;
                        lookup_word<0>(wq.x, lb, se, so);
                        lookup_word<1>(wq.y, lb, se, so);
                        lookup_word<2>(wq.z, lb, se, so);
                        lookup_word<3>(wq.w, lb, se, so);
                        acc[h * kLutUnitRows + rr] = ncur[h * kLutUnitRows + rr] * (se + so);
                    }
                }
                // the group's eight row sums
                const float v = reduce_rows8(acc, lane);
                const int k = (lane >> 2) & 7;
                const int64_t row = (g0 + (int64_t)i * gstride) * kRows + k;
                if ((lane & 3) == 0 && row < p.N) {
                    if (p.nranges == 1) {
                        p.Y[(int64_t)p.t * p.N + row] = v * yscale;
                    } else {
                        float* pp = part + (w + i * kLutWarps) * kRows + k;
                        *pp = (r == 0) ? v : *pp + v;
                    }
                }
            }
            u_glob += nunits;
        }
        if (p.nranges > 1) {   // this warp's rows of the block are final
            __syncwarp();
            for (int idx = lane; idx < ngw * kRows; idx += 32) {
                const int i = idx / kRows, k = idx % kRows;
                const int64_t row = (g0 + (int64_t)i * gstride) * kRows + k;
                if (row < p.N) p.Y[(int64_t)p.t * p.N + row] = part[(w + i * kLutWarps) * kRows + k] * yscale;
            }
            __syncwarp();
        }
    }
}

template <int F>
cq_status run_lut(LutParams p, int64_t B, cudaStream_t st) {
    static bool attr[64] = {};
    static std::mutex mu;
    auto kern = cq_gemv_lut_kernel<F>;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return check_launch();
    if (dev < 0 || dev >= 64) return CQ_ERR_UNSUPPORTED;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!attr[dev]) {
            if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kLutSmem) !=
                cudaSuccess)
                return check_launch();
            attr[dev] = true;
        }
    }
    p.smem_bytes = (uint32_t)kLutSmem;
    const int64_t ngroups = (p.N + kRows - 1) / kRows;
    int64_t grid = sm_count();
    if (ngroups < grid) grid = ngroups;
    p.groups_base = ngroups / grid;
    p.groups_extra = (int)(ngroups % grid);
    for (int64_t t = 0; t < B; ++t) {
        p.t = (int)t;
        const cq_status s = launch_pdl(kern, dim3((unsigned)grid), dim3(kLutThreads), kLutSmem, st, p);
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
    // the tensor copies address rows with 32-bit coordinates
    if (K > (1 << 24) || N > ((int64_t)1 << 31) - 64 || B > (1 << 30)) return CQ_ERR_UNSUPPORTED;
    if (!aligned16(packed) || !aligned16(norms) || !aligned16(Xq) || !aligned16(scale) || !aligned16(Y))
        return CQ_ERR_ALIGNMENT;
    LutParams p;
    p.norms = norms; p.Xq = Xq; p.scale = scale; p.Y = Y;
    {
        unsigned int* err = nullptr;
        const cq_status se = pipe::device_error_word(&err);
        if (se != CQ_OK) return se;
        p.err = err;
    }
    p.N = N; p.K = (int)K;
    const int f = cq_field_bits(b);
    p.words = (int)(K * f / 32);
    p.nranges = (p.words + kRangeWords - 1) / kRangeWords;
    p.groups_base = 0;
    p.groups_extra = 0;
    p.t = 0;
    p.smem_bytes = 0;
    {
        const uint64_t rowbytes = (uint64_t)p.words * 4u;
        const cq_status se = pipe::encode_map(&p.pmap, CU_TENSOR_MAP_DATA_TYPE_UINT32, packed, (uint64_t)p.words,
                                              (uint64_t)N, rowbytes, kRangeWords, kLutUnitRows);
        if (se != CQ_OK) return se;
    }
    float lv[16];
    cq_host_levels(lv, b, cbk);
    for (int u = 0; u < 4; ++u) p.lv[u] = lv[u];
    cudaStream_t st = as_stream(stream);
    return f == 1 ? run_lut<1>(p, B, st) : run_lut<2>(p, B, st);
}
