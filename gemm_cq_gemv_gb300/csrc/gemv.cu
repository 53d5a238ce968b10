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

#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "gemv_pipe.cuh"

namespace cq {
namespace {

using namespace pipe;

constexpr int kThreads = 256;   // 8 warps
constexpr int kSeg = 1024;      // positions per segment (32 lanes x 32)

// ---------------------------------------------------------------------------------
// A4: xr = Hu @ q per 128-group (Needle .cact page, §一, with H = Hu / sqrt(128) and
// H = H^T).  One warp per (token, group); values are small integers, exact in fp32.
// ---------------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads)
rotate_act_kernel(const int8_t* __restrict__ Xq, int64_t groups, float* __restrict__ xr) {
    pdl_trigger();
    pdl_wait();
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


// ---------------------------------------------------------------------------------
// Shared pieces of the two GEMV kernels.
//
// One CTA of 16 warps per SM, persistent over row tiles.  Warp w owns K-segment slots
// (w mod nsl) - plus slot + 16 when K has more than 16 segments - so its activation
// slice is loaded into registers once per kernel; when K has fewer segments than warps
// the warps sharing a segment split the tile into row groups of 8.  Every tile therefore
// needs a cross-warp sum: each warp drops its per-row partials into one of kSlots
// shared slots and counts itself in with an atomic add on the slot's counter; the warp
// that arrives last adds the partials in warp order (deterministic), writes the rows
// and frees the slot.  A warp waits only when it runs kSlots tiles ahead of the slowest
// one, so no warp stalls the streaming of the others.
// ---------------------------------------------------------------------------------
constexpr int kWarps2 = 16;


// ---------------------------------------------------------------------------------
// Per-warp staging ring.  Each warp streams its own rows through kRing slots of shared
// memory, one slot per unit of kUnitRows rows (half a warp tile) of one owned segment,
// filled by one 2-D tensor copy (cp.async.bulk.tensor, issued by one lane) that
// completes on the slot's mbarrier.  While a unit is decoded the next kRing - 1 are in
// flight, so the load latency overlaps the decode instead of following it.
// ---------------------------------------------------------------------------------
constexpr int kUnitRows = 4;
// smallest batch that cq_gemv sends to the tensor-core path (4-bit indices)
constexpr int64_t kTensorMinBatch = 3;
// row coordinates of the tensor copies are 32-bit (with a tile of slack past N)
constexpr int64_t kMaxGemvRows = ((int64_t)1 << 31) - 1024;
constexpr int kRing = 4;       // a power of two (slot = unit & 3, phase = unit >> 2)
static_assert(kRing == 4, "ring slot and phase arithmetic assume 4 slots");


// ---------------------------------------------------------------------------------
// A5: CQ GEMV.  Y[t][o] = s_t / 128 * sum_j norm[o][j] * sum_i cb[idx] * xr[t][128 j + i]
// Codewords come from a shared-memory table indexed by two consecutive indices (2b
// bits): entry e = (cb[e mod 2^b], cb[e / 2^b]), replicated once per bank so every lane
// reads its own copy (conflict-free 64-bit loads); the pair multiplies a pair of
// activations with two scalar FMAs.  For 4-bit indices the table sits at a 64 KB
// boundary of the shared window, so the address of (entry e, lane l), base | e << 8 |
// l << 3, is one byte permute of an index byte into the lane's base.  The packed rows
// and their group norms arrive through the warp's staging ring.
// ---------------------------------------------------------------------------------
struct CqGemvParams {
    CUtensorMap pmap;     // packed rows as [N][rowbytes / 4] uint32, box 32 b x kUnitRows
    CUtensorMap nmap;     // norms as [N][K / 128] fp16, box 8 x kUnitRows (when K % 1024 == 0)
    const uint8_t* packed;
    const uint16_t* norms;
    const float* xr;      // [B][K] rotated activations (multi-pass calls), or
    const int8_t* xq;     // [B][K] int8 activations, rotated in the prologue (single pass)
    const float* scale;   // [B]
    float* Y;             // [B][N]
    unsigned int* err;    // device error flag
    int64_t N;
    int K;
    int nseg;             // ceil(K / 1024)
    int rg;               // row groups per tile
    int t0;               // first token of this pass
    int ntok;             // tokens in this pass (<= TB)
    uint32_t smem_bytes;  // dynamic shared memory of the launch
    float lv[16];
};

template <int NB>
__device__ __forceinline__ uint32_t extract_bits(const uint32_t* w, int p) {
    // bits [NB p, NB p + NB) of the little-endian word string w
    const int pos = NB * p;
    const int wi = pos >> 5, sh = pos & 31;
    uint32_t v = w[wi] >> sh;
    if (sh + NB > 32) v |= w[wi + 1] << (32 - sh);
    return v & ((1u << NB) - 1u);
}

// this lane's 4 b bytes of a staged row segment
template <int BITS>
__device__ __forceinline__ void lds_packed(uint32_t (&w)[BITS], const uint8_t* p) {
    if constexpr (BITS == 4) {
        const uint4 v = *reinterpret_cast<const uint4*>(p);
        w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
    } else if constexpr (BITS == 2) {
        const uint2 v = *reinterpret_cast<const uint2*>(p);
        w[0] = v.x; w[1] = v.y;
    } else {
#pragma unroll
        for (int k = 0; k < BITS; ++k) w[k] = reinterpret_cast<const uint32_t*>(p)[k];
    }
}

template <int J>
__device__ __forceinline__ uint32_t pair_addr(uint32_t wv, uint32_t lb) {
    uint32_t a;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(a) : "r"(wv), "r"(lb), "n"(0x7604 | (J << 4)));
    return a;
}
__device__ __forceinline__ float2 lds_f2(uint32_t addr) {
    float2 v;
    asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr));
    return v;
}

// Shared-memory plan of the CQ kernel: pair table, reduction area, ring barriers and one
// ring per warp (a slot holds the kUnitRows x segment box of packed rows, then the
// kUnitRows x 8 box of their group norms; slots are 128-byte aligned for the copies).
template <int BITS>
struct CqPlan {
    static constexpr uint32_t seg = 128 * BITS;                        // bytes of a row segment
    static constexpr uint32_t norms = kUnitRows * seg;                  // offset of the norm box
    static constexpr uint32_t slot = (norms + kUnitRows * 16 + 127) / 128 * 128;
    static constexpr uint32_t ring = kRing * slot;
    static constexpr uint32_t table = (1u << (2 * BITS)) * 32 * 8;
};

template <int BITS>
size_t cq_smem_bytes(int tb) {
    using P = CqPlan<BITS>;
    const size_t rest = reduce_bytes<kWarps2>(tb) + 16 + kWarps2 * kRing * 8 + 8 + 64 + 16 +
                        (size_t)kWarps2 * (P::ring + 128);
    // 4-bit: the table is 64 KB aligned; the space below it may be too small to use
    if (BITS == 4) return 227 * 1024;
    return P::table + 16 + rest;
}

// xr = Hu @ q for this lane's 32 positions of a 128-group held by lanes 4g..4g+3: five
// butterfly stages inside the lane, the strides of 32 and 64 across lanes (xor 1, 2).
// The values are integers below 2^24, exact in fp32 in any order, so this equals the
// separate rotation kernel bit for bit.
__device__ __forceinline__ void rotate32(float (&v)[32], int lane) {
#pragma unroll
    for (int h = 1; h < 32; h <<= 1)
#pragma unroll
        for (int j = 0; j < 32; ++j)
            if ((j & h) == 0) {
                const float a = v[j], b = v[j + h];
                v[j] = a + b;
                v[j + h] = a - b;
            }
#pragma unroll
    for (int m = 1; m <= 2; m <<= 1) {
        const bool upper = (lane & m) != 0;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const float q = __shfl_xor_sync(0xffffffffu, v[j], m);
            v[j] = upper ? (q - v[j]) : (v[j] + q);
        }
    }
}

template <int BITS, int TB, int SPW>
__global__ void __launch_bounds__(kWarps2 * 32, 1) cq_gemv_kernel(const __grid_constant__ CqGemvParams p) {
    using P = CqPlan<BITS>;
    constexpr int L = 1 << BITS;
    constexpr int E = 1 << (2 * BITS);
    extern __shared__ __align__(128) unsigned char smem_c[];
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    pdl_trigger();
    const uint32_t sbase = smem_u32(smem_c), send = sbase + p.smem_bytes;
    uint32_t tbase;
    SmemCarve cv;
    cv.ok = true;
    if (BITS == 4) {
        tbase = (sbase + 65535u) & ~65535u;
        cv.a = sbase; cv.a_end = tbase; cv.b = tbase + P::table; cv.b_end = send;
    } else {
        tbase = (sbase + 15u) & ~15u;
        cv.a = cv.a_end = tbase + P::table; cv.b = cv.a; cv.b_end = send;
    }
    if (tbase + P::table > send) cv.ok = false;
    const uint32_t red_at = cv.take((uint32_t)reduce_bytes<kWarps2>(TB), 16);
    const uint32_t bar_at = cv.take(kWarps2 * kRing * 8, 8);
    const uint32_t lv_at = cv.take(16 * sizeof(float), 16);
    uint32_t ring_at = 0;
    for (int v = 0; v < kWarps2; ++v) {
        const uint32_t at = cv.take(P::ring, 128);
        if (v == w) ring_at = at;
    }
    if (!cv.ok) {   // the launch's shared memory cannot hold the plan (host sizing error)
        if (tid == 0) atomicOr(p.err, 4u);
        return;
    }
    auto gen = [&](uint32_t a) { return smem_c + (a - sbase); };
    float2* lut2 = reinterpret_cast<float2*>(gen(tbase));                 // [E][32]
    const Reduce rd = carve_reduce<kWarps2>(gen(red_at), TB);
    uint64_t* rfull = reinterpret_cast<uint64_t*>(gen(bar_at)) + w * kRing;
    float* slv = reinterpret_cast<float*>(gen(lv_at));
    uint8_t* ring = gen(ring_at);
    if (tid == 0) {
        prefetch_tensormap(&p.pmap);
        if (p.K % kSeg == 0) prefetch_tensormap(&p.nmap);
    }
    if (lane < kRing) mbar_init(&rfull[lane], 1);   // each warp its own ring barriers
    if (tid < kSlots) {
        rd.count[tid] = 0u;
        mbar_init(&rd.empty[tid], 1);
    }
    if (lane == 0) asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    if (tid < 16) {   // the levels, by an unrolled select (no indexed parameter access)
        float v = 0.0f;
#pragma unroll
        for (int u = 0; u < 16; ++u) v = (u == tid) ? p.lv[u] : v;
        slv[tid] = v;
    }
    __syncthreads();

    const int nsl = p.nseg < kWarps2 ? p.nseg : kWarps2;
    const int slot = w % nsl, rgi = w / nsl;
    const uint32_t nbusy = (uint32_t)(nsl * p.rg);
    const bool busy = rgi < p.rg;
    const int G = p.K / kGroup;
    const int tile_rows = kRows * p.rg;
    const int64_t ntiles = (p.N + tile_rows - 1) / tile_rows;
    const int64_t ntk = (int64_t)blockIdx.x < ntiles ? (ntiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    const int nown = (SPW == 2 && slot + kWarps2 < p.nseg) ? 2 : 1;   // owned segments
    const int upt = 2 * nown;                                           // units per tile
    const int64_t U = busy ? ntk * upt : 0;
    const bool nbulk = (p.K % kSeg) == 0;   // a segment's norms are 16 aligned bytes

    // cursor of the next unit to issue (units go out strictly in order)
    int64_t nx_base = (int64_t)blockIdx.x * tile_rows + (int64_t)rgi * kRows;   // its tile's first row
    int nx_rem = 0;                                                             // unit within the tile
    constexpr uint32_t kBoxBytes = kUnitRows * P::seg;
    auto issue = [&](int d) {
        if (lane == 0) {
            const int seg = slot + (nx_rem >> 1) * kWarps2;
            const int y = (int)(nx_base + (nx_rem & 1) * kUnitRows);
            uint8_t* sp = ring + d * P::slot;
            mbar_arrive_tx(&rfull[d], kBoxBytes + (nbulk ? kUnitRows * 16u : 0u));
            tma_box(sp, &p.pmap, seg * (P::seg / 4), y, &rfull[d]);
            if (nbulk) tma_box(sp + P::norms, &p.nmap, seg * 8, y, &rfull[d]);
        }
        if (++nx_rem == upt) {
            nx_rem = 0;
            nx_base += (int64_t)gridDim.x * tile_rows;
        }
    };
    // the table is built while the previous kernel of the stream finishes; then the
    // first units go in flight while the activations are set up
    for (int i = tid; i < E * 32; i += kWarps2 * 32) {
        const int e = i >> 5;
        lut2[i] = make_float2(slv[e & (L - 1)], slv[e >> BITS]);
    }
    pdl_wait();
    for (int64_t u = 0; u < kRing - 1 && u < U; ++u) issue((int)u);
    float2 xx[SPW][TB][16];
#pragma unroll
    for (int i = 0; i < SPW; ++i) {
        const int seg = slot + i * kWarps2;
        const int pos0 = seg * kSeg + lane * 32;
#pragma unroll
        for (int t = 0; t < TB; ++t) {
            // whole 128-groups lie inside or outside K, so the four lanes of a group agree
            const bool ok = busy && seg < p.nseg && pos0 < p.K && t < p.ntok;
            if (p.xq) {
                float v[32];
                const int8_t* src = p.xq + (int64_t)(p.t0 + t) * p.K + pos0;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int4 c = ok ? *reinterpret_cast<const int4*>(src + 16 * h) : make_int4(0, 0, 0, 0);
                    const int wv[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
                    for (int q = 0; q < 16; ++q) v[16 * h + q] = (float)(int8_t)(wv[q >> 2] >> (8 * (q & 3)));
                }
                rotate32(v, lane);
#pragma unroll
                for (int q = 0; q < 16; ++q) xx[i][t][q] = make_float2(v[2 * q], v[2 * q + 1]);
            } else {
                const float* src = p.xr + (int64_t)(p.t0 + t) * p.K + pos0;
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const float4 v = ok ? *reinterpret_cast<const float4*>(src + 4 * q)
                                        : make_float4(0.f, 0.f, 0.f, 0.f);
                    xx[i][t][2 * q] = make_float2(v.x, v.y);
                    xx[i][t][2 * q + 1] = make_float2(v.z, v.w);
                }
            }
        }
    }
    __syncthreads();
    if (!busy) return;   // warps left over when the segments do not divide 16

    const float2* mylut = lut2 + lane;
    const uint32_t lb = tbase | ((uint32_t)lane << 3);
    int64_t u = 0;
    for (int64_t k = 0; k < ntk; ++k) {
        const int64_t tile = blockIdx.x + k * gridDim.x;
        float acc[TB][kRows];
#pragma unroll
        for (int t = 0; t < TB; ++t)
#pragma unroll
            for (int r = 0; r < kRows; ++r) acc[t][r] = 0.0f;
#pragma unroll
        for (int i = 0; i < SPW; ++i) {
            if (i >= nown) break;
            const int seg = slot + i * kWarps2;
            const bool active = seg * kSeg + lane * 32 < p.K;
#pragma unroll
            for (int h = 0; h < 2; ++h, ++u) {
                if (u + kRing - 1 < U) {
                    fence_proxy_async();   // reads of the slot about to be refilled are done
                    __syncwarp();
                    issue((int)((u + kRing - 1) & (kRing - 1)));
                }
                const int64_t row0 = tile * tile_rows + (int64_t)rgi * kRows + h * kUnitRows;
                const int64_t left = p.N - row0;
                const int nv = !active ? 0 : (left >= kUnitRows ? kUnitRows : (int)left);   // rows to add
                const int d = (int)(u & (kRing - 1));
                const uint8_t* sp = ring + d * P::slot;
                float nrm[kUnitRows];
                if (!nbulk) {
#pragma unroll
                    for (int r = 0; r < kUnitRows; ++r)
                        nrm[r] = r < nv ? f16_bits_to_f32(__ldg(p.norms + (row0 + r) * G + seg * 8 + (lane >> 2)))
                                        : 0.0f;
                }
                mbar_wait(&rfull[d], (uint32_t)(u >> 2) & 1u, p.err);
                if (nbulk) {
                    const uint16_t* sn = reinterpret_cast<const uint16_t*>(sp + P::norms);
#pragma unroll
                    for (int r = 0; r < kUnitRows; ++r)
                        nrm[r] = r < nv ? f16_bits_to_f32(sn[r * 8 + (lane >> 2)]) : 0.0f;
                }
#pragma unroll
                for (int r = 0; r < kUnitRows; ++r) {
                    uint32_t wd[BITS];
                    lds_packed<BITS>(wd, sp + r * P::seg + lane * (4 * BITS));
                    // scalar FMAs on four independent chains per token: the FMA pipe has room,
                    // the integer pipe (byte permutes, moves) is the one that binds
                    float a4[TB][4];
#pragma unroll
                    for (int t = 0; t < TB; ++t) a4[t][0] = a4[t][1] = a4[t][2] = a4[t][3] = 0.0f;
                    if constexpr (BITS == 4) {
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            const uint32_t wv = wd[kk];
                            const float2 c0 = lds_f2(pair_addr<0>(wv, lb));
                            const float2 c1 = lds_f2(pair_addr<1>(wv, lb));
                            const float2 c2 = lds_f2(pair_addr<2>(wv, lb));
                            const float2 c3 = lds_f2(pair_addr<3>(wv, lb));
#pragma unroll
                            for (int t = 0; t < TB; ++t) {
                                const float2* xq = &xx[i][t][4 * kk];
                                a4[t][0] = fmaf(c0.x, xq[0].x, a4[t][0]); a4[t][1] = fmaf(c0.y, xq[0].y, a4[t][1]);
                                a4[t][2] = fmaf(c1.x, xq[1].x, a4[t][2]); a4[t][3] = fmaf(c1.y, xq[1].y, a4[t][3]);
                                a4[t][0] = fmaf(c2.x, xq[2].x, a4[t][0]); a4[t][1] = fmaf(c2.y, xq[2].y, a4[t][1]);
                                a4[t][2] = fmaf(c3.x, xq[3].x, a4[t][2]); a4[t][3] = fmaf(c3.y, xq[3].y, a4[t][3]);
                            }
                        }
                    } else {
#pragma unroll
                        for (int q = 0; q < 16; ++q) {
                            const float2 c = mylut[extract_bits<2 * BITS>(wd, q) << 5];
#pragma unroll
                            for (int t = 0; t < TB; ++t) {
                                a4[t][2 * (q & 1)] = fmaf(c.x, xx[i][t][q].x, a4[t][2 * (q & 1)]);
                                a4[t][2 * (q & 1) + 1] = fmaf(c.y, xx[i][t][q].y, a4[t][2 * (q & 1) + 1]);
                            }
                        }
                    }
#pragma unroll
                    for (int t = 0; t < TB; ++t)
                        acc[t][h * kUnitRows + r] =
                            fmaf(nrm[r], (a4[t][0] + a4[t][2]) + (a4[t][1] + a4[t][3]), acc[t][h * kUnitRows + r]);
                }
            }
        }
        tile_reduce<TB, kWarps2>(rd, acc, (int)k, w, lane, nsl, nbusy, tile_rows, p.ntok, p.err,
                        [&](int t, int rr, float sum) {
                            const int64_t row = tile * tile_rows + rr;
                            if (row < p.N) {
                                const int tok = p.t0 + t;
                                p.Y[(int64_t)tok * p.N + row] = sum * (p.scale[tok] * (1.0f / 128.0f));
                            }
                        });
    }
}

// ---------------------------------------------------------------------------------
// A8: Q4_0 GEMV.  Same persistent layout; lane l of a segment owns block 32 seg + l of
// every row.  The 18-byte blocks of a row segment are staged in shared memory - through
// the warp's ring when rows and segments are 16-byte aligned, else by guarded 16-byte
// loads into one buffer per warp - and each lane reads its block with five aligned
// 32-bit loads.  The lane's activations of a block become 24-bit fixed-point integers
// once (q4_fix), split into three byte planes; a block then costs, per packed word of
// eight nibbles, two masks and six dp4a (nibble bytes times activation bytes, exact in
// int32), and one scale per block.
// ---------------------------------------------------------------------------------
struct Q40GemvParams {
    CUtensorMap bmap;     // blocks as [N][nblk * 18 / 4] uint32, box 144 x kUnitRows (nblk % 8 == 0)
    const uint8_t* blocks;
    const float* X;       // [B][K]
    float* Y;             // [B][N]
    unsigned int* err;
    int64_t N;
    int K;
    int nblk;             // ceil(K / 32)
    int nseg;             // ceil(nblk / 32)
    int rg;
    int64_t total_bytes;  // N * nblk * 18
    int t0, ntok;
    int64_t groups_base;  // ring kernel: a CTA takes groups_base row groups (8 rows), one
    int groups_extra;     //   more if blockIdx.x < groups_extra
};

constexpr int kStage = 608;     // >= 37 chunks of 16 B, per row (unaligned staging)
constexpr int kQSeg = 576;      // 32 blocks of 18 B (ring staging)

// A lane's 32 activations of one block as a 24-bit fixed-point integer per position,
// X_i = rint(x_i * 2^e) with 2^e the power of two that brings the block's largest |x|
// into [2^21, 2^22): the rounding error is at most 2^-23 of that largest value, the
// precision of an fp32 mantissa.  X_i = X0_i + 256 X1_i + 65536 X2_i (bytes X0, X1
// unsigned, X2 signed); plane p packs byte p of the even positions 8k, 8k+2, 8k+4, 8k+6
// (e[p][k]) and of the odd ones (o[p][k]) in the order of the nibbles of packed word k.
struct Q4X {
    uint32_t e[3][4], o[3][4];
    int c[3];      // 8 * sum_i plane_p(X_i): the -8 of the format, per plane
    float inv;     // 2^-e (NaN when the block holds a non-finite activation)
};

__device__ __forceinline__ int dp4a_uu(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ int dp4a_su(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
// byte P of a, b, c, d -> bytes 0..3
template <int P>
__device__ __forceinline__ uint32_t pack_bytes(uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    uint32_t lo, hi, r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(lo) : "r"(a), "r"(b), "n"(P | ((4 + P) << 4)));
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(hi) : "r"(c), "r"(d), "n"(P | ((4 + P) << 4)));
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(lo), "r"(hi), "n"(0x5410));
    return r;
}

__device__ __forceinline__ void q4_fix(const float (&x)[32], Q4X& q) {
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        float a;
        asm("max.NaN.f32 %0, %1, %2;" : "=f"(a) : "f"(amax), "f"(fabsf(x[i])));
        amax = a;
    }
    int E = (int)(__float_as_uint(amax) >> 23);   // amax < 2^(E - 126)
    const bool finite = E < 255;
    if (E < 22) E = 22;                            // zero or tiny blocks
    if (E > 254) E = 254;
    const float sc = __uint_as_float((uint32_t)(275 - E) << 23);    // 2^(148 - E)
    q.inv = finite ? __uint_as_float((uint32_t)(E - 21) << 23) : __uint_as_float(0x7fc00000u);
    uint32_t X[32];
#pragma unroll
    for (int i = 0; i < 32; ++i)   // |x sc| < 2^22: 1.5 * 2^23 + x sc rounds x sc to an integer
        X[i] = (uint32_t)(__float_as_int(fmaf(x[i], sc, 12582912.0f)) - 0x4B400000);
    int c0 = 0, c1 = 0, c2 = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        q.e[0][k] = pack_bytes<0>(X[8 * k], X[8 * k + 2], X[8 * k + 4], X[8 * k + 6]);
        q.o[0][k] = pack_bytes<0>(X[8 * k + 1], X[8 * k + 3], X[8 * k + 5], X[8 * k + 7]);
        q.e[1][k] = pack_bytes<1>(X[8 * k], X[8 * k + 2], X[8 * k + 4], X[8 * k + 6]);
        q.o[1][k] = pack_bytes<1>(X[8 * k + 1], X[8 * k + 3], X[8 * k + 5], X[8 * k + 7]);
        q.e[2][k] = pack_bytes<2>(X[8 * k], X[8 * k + 2], X[8 * k + 4], X[8 * k + 6]);
        q.o[2][k] = pack_bytes<2>(X[8 * k + 1], X[8 * k + 3], X[8 * k + 5], X[8 * k + 7]);
        c0 = dp4a_uu(q.e[0][k], 0x01010101u, dp4a_uu(q.o[0][k], 0x01010101u, c0));
        c1 = dp4a_uu(q.e[1][k], 0x01010101u, dp4a_uu(q.o[1][k], 0x01010101u, c1));
        c2 = dp4a_su(q.e[2][k], 0x01010101u, dp4a_su(q.o[2][k], 0x01010101u, c2));
    }
    q.c[0] = 8 * c0;
    q.c[1] = 8 * c1;
    q.c[2] = 8 * c2;
}

// One 18-byte block of a row against the fixed-point activations:
//   sum_i (nib_i - 8) x_i = 2^-e * sum_p 256^p (sum_i nib_i Xp_i - 8 sum_i Xp_i),
// each plane's sum exact in int32 (dp4a of the nibble bytes and the activation bytes).
// A block of nibbles all 8 (every weight 0, e.g. an all-zero row: KMCU page, §2) gives
// exactly 0.
template <int TB>
__device__ __forceinline__ void q4_block(const uint32_t* wp, uint32_t dsh, uint32_t nsh,
                                         const Q4X (&xq)[TB], float (&acc)[TB][kRows], int r) {
    // wp: the aligned words covering the block; dsh: bit offset of the fp16 scale in
    // word 0 (0 or 16); nsh = dsh + 16: funnel shift that aligns the nibble bytes
    const uint32_t w0 = wp[0], w1 = wp[1], w2 = wp[2], w3 = wp[3], w4 = wp[4];
    const float d = f16_bits_to_f32((uint16_t)(w0 >> dsh));
    const uint32_t nw[4] = {__funnelshift_rc(w0, w1, nsh), __funnelshift_rc(w1, w2, nsh),
                            __funnelshift_rc(w2, w3, nsh), __funnelshift_rc(w3, w4, nsh)};
    int s0[TB], s1[TB], s2[TB];
#pragma unroll
    for (int t = 0; t < TB; ++t) s0[t] = s1[t] = s2[t] = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        // even-index nibbles (low halves of the bytes) and odd-index nibbles, one per byte
        const uint32_t ev = nw[k] & 0x0F0F0F0Fu, od = (nw[k] >> 4) & 0x0F0F0F0Fu;
#pragma unroll
        for (int t = 0; t < TB; ++t) {
            s0[t] = dp4a_uu(ev, xq[t].e[0][k], s0[t]);
            s0[t] = dp4a_uu(od, xq[t].o[0][k], s0[t]);
            s1[t] = dp4a_uu(ev, xq[t].e[1][k], s1[t]);
            s1[t] = dp4a_uu(od, xq[t].o[1][k], s1[t]);
            s2[t] = dp4a_us(ev, xq[t].e[2][k], s2[t]);
            s2[t] = dp4a_us(od, xq[t].o[2][k], s2[t]);
        }
    }
#pragma unroll
    for (int t = 0; t < TB; ++t) {
        // |s0 - c0| < 2^17 and |s1 - c1| < 2^17: the low two planes in int32
        const int lo = (s0[t] - xq[t].c[0]) + 256 * (s1[t] - xq[t].c[1]);
        const float v = fmaf(65536.0f, (float)(s2[t] - xq[t].c[2]), (float)lo);
        acc[t][r] = fmaf(d * xq[t].inv, v, acc[t][r]);
    }
}

// This lane's blocks of activations (zero outside K) in fixed point; 16-byte loads where
// the block lies inside K and rows of X are 16-byte aligned.
template <int TB, int SPW>
__device__ __forceinline__ void q4_load_x(const Q40GemvParams& p, int slot, bool busy, int lane,
                                          Q4X (&xq)[SPW][TB]) {
#pragma unroll
    for (int i = 0; i < SPW; ++i) {
        const int seg = slot + i * kWarps2;
        const int blk = seg * 32 + lane;
#pragma unroll
        for (int t = 0; t < TB; ++t) {
            const bool ok = busy && seg < p.nseg && blk < p.nblk && t < p.ntok;
            const float* src = p.X + (int64_t)(p.t0 + t) * p.K + blk * 32;
            float x[32];
            if (ok && (p.K & 3) == 0 && blk * 32 + 32 <= p.K) {
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const float4 v = __ldg(reinterpret_cast<const float4*>(src) + q);
                    x[4 * q] = v.x; x[4 * q + 1] = v.y; x[4 * q + 2] = v.z; x[4 * q + 3] = v.w;
                }
            } else {
#pragma unroll
                for (int q = 0; q < 32; ++q) x[q] = (ok && blk * 32 + q < p.K) ? src[q] : 0.0f;
            }
            q4_fix(x, xq[i][t]);
        }
    }
}

// Ring-staged Q4_0 GEMV: needs 16-byte aligned row segments (nblk a multiple of 8).
template <int TB, int SPW>
__global__ void __launch_bounds__(kWarps2 * 32, 1) q4_0_gemv_ring_kernel(const __grid_constant__ Q40GemvParams p) {
    extern __shared__ __align__(128) uint8_t smem_q[];
    constexpr int kSlotB = kUnitRows * kQSeg;
    uint8_t* rings = smem_q;                                                   // [16][kRing][4][576]
    uint64_t* rbar = reinterpret_cast<uint64_t*>(smem_q + kWarps2 * kRing * kSlotB);  // [16][kRing]
    const Reduce rd = carve_reduce_sets<kWarps2>(rbar + kWarps2 * kRing, TB, kWarps2);
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    pdl_trigger();
    const int nsl = p.nseg < kWarps2 ? p.nseg : kWarps2;
    const int slot = w % nsl, rgi = w / nsl;
    const bool busy = rgi < p.rg;
    uint8_t* ring = rings + w * (kRing * kSlotB);
    uint64_t* rfull = rbar + w * kRing;
    // a warp's ring barriers are its own: it initialises them and starts its first copies
    // at once; the activations are converted while those copies are in flight
    if (tid == 0) prefetch_tensormap(&p.bmap);
    if (lane < kRing) mbar_init(&rfull[lane], 1);
    for (int i = tid; i < p.rg * kSlots; i += kWarps2 * 32) {
        rd.count[i] = 0u;
        mbar_init(&rd.empty[i], 1);
    }
    if (lane == 0) asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    __syncwarp();

    // row group j (8 rows) belongs to CTA j mod G; the CTA's m-th group goes to warp set
    // m mod rg (the nsl warps sharing a row group, one per segment)
    const int64_t ncta = p.groups_base + ((int)blockIdx.x < p.groups_extra ? 1 : 0);
    const int64_t ngr = busy && ncta > rgi ? (ncta - rgi + p.rg - 1) / p.rg : 0;
    const int64_t gstep = (int64_t)kRows * p.rg * gridDim.x;
    const int64_t row0 = (int64_t)kRows * (blockIdx.x + (int64_t)rgi * gridDim.x);
    const int nown = (SPW == 2 && slot + kWarps2 < p.nseg) ? 2 : 1;
    const int upt = 2 * nown;
    const int64_t U = ngr * upt;

    int64_t nx_base = row0;
    int nx_rem = 0;
    auto issue = [&](int d) {
        if (lane == 0) {
            const int seg = slot + (nx_rem >> 1) * kWarps2;
            const int y = (int)(nx_base + (nx_rem & 1) * kUnitRows);
            mbar_arrive_tx(&rfull[d], (uint32_t)kSlotB);
            tma_box(ring + d * kSlotB, &p.bmap, seg * (kQSeg / 4), y, &rfull[d]);
        }
        if (++nx_rem == upt) {
            nx_rem = 0;
            nx_base += gstep;
        }
    };
    // the weight blocks are read before the wait for the previous kernel of the stream
    // (weights come from kernels that release their dependents only at completion), the
    // activations after it
    for (int64_t u = 0; u < kRing - 1 && u < U; ++u) issue((int)u);
    pdl_wait();
    Q4X xq[SPW][TB];
    q4_load_x<TB, SPW>(p, slot, busy, lane, xq);
    __syncthreads();   // every warp set's reduction barriers initialised
    if (!busy) return;   // warps left over when the segments do not divide 16

    // every staged row starts at byte 0: per-lane word offset and shifts
    const int o = lane * 18;
    const uint32_t dsh = (uint32_t)(o & 3) * 8u;
    int64_t u = 0;
    for (int64_t k = 0; k < ngr; ++k) {
        const int64_t rbase = row0 + k * gstep;   // the group's first row
        float acc[TB][kRows];
#pragma unroll
        for (int t = 0; t < TB; ++t)
#pragma unroll
            for (int r = 0; r < kRows; ++r) acc[t][r] = 0.0f;
#pragma unroll
        for (int i = 0; i < SPW; ++i) {
            if (i >= nown) break;
#pragma unroll
            for (int h = 0; h < 2; ++h, ++u) {
                if (u + kRing - 1 < U) {
                    fence_proxy_async();   // reads of the slot about to be refilled are done
                    __syncwarp();
                    issue((int)((u + kRing - 1) & (kRing - 1)));
                }
                const int d = (int)(u & (kRing - 1));
                mbar_wait(&rfull[d], (uint32_t)(u >> 2) & 1u, p.err);
                const uint32_t* wl = reinterpret_cast<const uint32_t*>(ring + d * kSlotB) + (o >> 2);
                // all four rows unconditionally, so their chains interleave: rows past N and
                // blocks past the row's end arrive as zeros (scale 0, nothing added), and the
                // activations of blocks past K are zero
#pragma unroll
                for (int r = 0; r < kUnitRows; ++r)
                    q4_block<TB>(wl + r * (kQSeg / 4), dsh, dsh + 16u, xq[i], acc, h * kUnitRows + r);
            }
        }
        group_reduce<TB, kWarps2>(rd, acc, (int)k, w, lane, nsl, rgi, p.ntok, p.err,
                                  [&](int t, int r, float sum) {
                                      const int64_t row = rbase + r;
                                      if (row < p.N) p.Y[(int64_t)(p.t0 + t) * p.N + row] = sum;
                                  });
    }
}

// Q4_0 GEMV for rows that are not 16-byte aligned: guarded 16-byte loads into one
// staging buffer of kRows rows per warp.
template <int TB, int SPW>
__global__ void __launch_bounds__(kWarps2 * 32, 1) q4_0_gemv_rows_kernel(const Q40GemvParams p) {
    extern __shared__ __align__(128) uint8_t smem_q[];
    uint8_t* stage = smem_q;                                              // [16][8][608]
    const Reduce rd = carve_reduce<kWarps2>(smem_q + kWarps2 * kRows * kStage, TB);
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    pdl_trigger();
    if (tid == 0) init_reduce(rd);
    pdl_wait();
    const int nsl = p.nseg < kWarps2 ? p.nseg : kWarps2;
    const int slot = w % nsl, rgi = w / nsl;
    const bool busy = rgi < p.rg;
    const uint32_t nbusy = (uint32_t)(nsl * p.rg);
    Q4X xq[SPW][TB];
    q4_load_x<TB, SPW>(p, slot, busy, lane, xq);
    __syncthreads();
    if (!busy) return;

    uint8_t* mystage = stage + w * (kRows * kStage);
    const int64_t rowbytes = (int64_t)p.nblk * 18;
    const int tile_rows = kRows * p.rg;
    const int64_t ntiles = (p.N + tile_rows - 1) / tile_rows;
    const uintptr_t base_addr = reinterpret_cast<uintptr_t>(p.blocks);
    const uintptr_t end_addr = base_addr + (uintptr_t)p.total_bytes;
    int it = 0;
    for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++it) {
        const int64_t row0 = tile * tile_rows + (int64_t)rgi * kRows;
        float acc[TB][kRows];
#pragma unroll
        for (int t = 0; t < TB; ++t)
#pragma unroll
            for (int r = 0; r < kRows; ++r) acc[t][r] = 0.0f;
#pragma unroll
        for (int i = 0; i < SPW; ++i) {
            const int seg = slot + i * kWarps2;
            if (seg >= p.nseg) break;
            const int nb = min(32, p.nblk - seg * 32);
            int offs[kRows];
            __syncwarp();
#pragma unroll
            for (int r = 0; r < kRows; ++r) {
                const int64_t row = row0 + r;
                offs[r] = 0;
                if (row >= p.N) continue;
                const uintptr_t a = base_addr + (uintptr_t)(row * rowbytes + (int64_t)seg * kQSeg);
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
                        for (int kk = 0; kk < 16; ++kk)
                            tmp[kk] = (q + kk < end_addr) ? *reinterpret_cast<const uint8_t*>(q + kk) : 0;
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
#pragma unroll
                for (int r = 0; r < kRows; ++r) {
                    if (row0 + r >= p.N) continue;
                    const int o = offs[r] + lane * 18;
                    const uint32_t dsh = (uint32_t)(o & 3) * 8u;
                    const uint32_t* wl = reinterpret_cast<const uint32_t*>(mystage + r * kStage) + (o >> 2);
                    q4_block<TB>(wl, dsh, dsh + 16u, xq[i], acc, r);
                }
            }
        }
        tile_reduce<TB, kWarps2>(rd, acc, it, w, lane, nsl, nbusy, tile_rows, p.ntok, p.err,
                        [&](int t, int rr, float sum) {
                            const int64_t row = tile * tile_rows + rr;
                            if (row < p.N) p.Y[(int64_t)(p.t0 + t) * p.N + row] = sum;
                        });
    }
}

constexpr size_t kMaxSmem = 227 * 1024;

static __device__ unsigned int g_gemv_err;
std::mutex g_err_mu;
unsigned int* g_gemv_err_ptr[64] = {nullptr};

}  // namespace

namespace pipe {
// Cached device address of this unit's error word on the current device.
cq_status device_error_word(unsigned int** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) { set_last_cuda_error((int)e); return CQ_ERR_CUDA; }
    if (dev < 0 || dev >= 64) return CQ_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_err_mu);
    if (!g_gemv_err_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_gemv_err);
        if (e != cudaSuccess) { set_last_cuda_error((int)e); return CQ_ERR_CUDA; }
        g_gemv_err_ptr[dev] = static_cast<unsigned int*>(p);
    }
    *out = g_gemv_err_ptr[dev];
    return CQ_OK;
}
}  // namespace pipe

namespace {

// Failure-detection probe: one thread waits, with this unit's bounded wait, on a barrier
// phase that nothing completes.  The wait gives up after `timeout_ns`, raises the error
// word and the kernel returns; nothing faults or hangs.
__global__ void bounded_wait_probe_kernel(unsigned int* err, unsigned long long timeout_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        mbar_wait(&bar, 0u, err, timeout_ns);
    }
}

}  // namespace

namespace pipe {
// cuTensorMapEncodeTiled from the driver (cached; no link against libcuda)
std::mutex g_enc_mu;
PFN_cuTensorMapEncodeTiled_v12000 g_enc = nullptr;

cq_status encode_map(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner,
                     uint64_t rows, uint64_t row_bytes, uint32_t box_inner, uint32_t box_rows) {
    {
        std::lock_guard<std::mutex> lock(g_enc_mu);
        if (!g_enc) {
            cudaDriverEntryPointQueryResult q;
            void* fn = nullptr;
            const cudaError_t e =
                cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
            if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) {
                set_last_cuda_error((int)e);
                return CQ_ERR_UNSUPPORTED;
            }
            g_enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        }
    }
    cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
    cuuint32_t box[2] = {box_inner, box_rows};
    cuuint32_t estr[2] = {1u, 1u};
    const CUresult r = g_enc(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) { set_last_cuda_error((int)r); return CQ_ERR_CUDA; }
    return CQ_OK;
}
}  // namespace pipe

namespace {

// `attr`: one flag per device (the shared-memory attribute is set per device context)
template <typename Kern>
cq_status launch_once(Kern kern, size_t smem, int64_t ntiles, cudaStream_t st, bool (&attr)[64],
                      int* grid_out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return check_launch();
    if (dev < 0 || dev >= 64) return CQ_ERR_UNSUPPORTED;
    if (!attr[dev]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kMaxSmem) !=
            cudaSuccess)
            return check_launch();
        attr[dev] = true;
    }
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kWarps2 * 32, smem) != cudaSuccess)
        return check_launch();
    if (per_sm < 1) return CQ_ERR_UNSUPPORTED;
    int64_t grid = (int64_t)per_sm * sm_count();
    if (ntiles < grid) grid = ntiles;
    *grid_out = (int)(grid < 1 ? 1 : grid);
    return CQ_OK;
}

// segment ownership: row groups when K has fewer segments than warps
inline int row_groups(int nseg) { return nseg >= kWarps2 ? 1 : kWarps2 / nseg; }

template <int BITS, int TB, int SPW>
cq_status run_cq_gemv(CqGemvParams p, cudaStream_t st) {
    static bool attr[64] = {};
    auto kern = cq_gemv_kernel<BITS, TB, SPW>;
    const size_t smem = cq_smem_bytes<BITS>(TB);
    p.smem_bytes = (uint32_t)smem;
    const int64_t ntiles = (p.N + (int64_t)kRows * p.rg - 1) / ((int64_t)kRows * p.rg);
    int grid = 0;
    const cq_status s = launch_once(kern, smem, ntiles, st, attr, &grid);
    if (s != CQ_OK) return s;
    return launch_pdl(kern, dim3(grid), dim3(kWarps2 * 32), smem, st, p);
}

template <int TB, int SPW, bool RING>
cq_status run_q4_0_gemv(Q40GemvParams p, cudaStream_t st) {
    static bool attr[64] = {};
    auto kern = RING ? q4_0_gemv_ring_kernel<TB, SPW> : q4_0_gemv_rows_kernel<TB, SPW>;
    const size_t smem = RING ? (size_t)kWarps2 * kRing * kUnitRows * kQSeg + kWarps2 * kRing * 8 +
                                   reduce_bytes_sets<kWarps2>(TB, kWarps2)
                             : (size_t)kWarps2 * kRows * kStage + reduce_bytes<kWarps2>(TB);
    // the ring kernel schedules row groups of 8 rows, the row-staged kernel tiles
    const int64_t nwork = RING ? (p.N + kRows - 1) / kRows
                               : (p.N + (int64_t)kRows * p.rg - 1) / ((int64_t)kRows * p.rg);
    int grid = 0;
    const cq_status s = launch_once(kern, smem, nwork, st, attr, &grid);
    if (s != CQ_OK) return s;
    p.groups_base = nwork / grid;
    p.groups_extra = (int)(nwork % grid);
    return launch_pdl(kern, dim3(grid), dim3(kWarps2 * 32), smem, st, p);
}

template <int BITS>
cq_status dispatch_cq(CqGemvParams p, int tb, int spw, cudaStream_t st) {
    if (spw == 2) return run_cq_gemv<BITS, 1, 2>(p, st);
    if (tb == 2) return run_cq_gemv<BITS, 2, 1>(p, st);
    return run_cq_gemv<BITS, 1, 1>(p, st);
}

}  // namespace

cq_status probe_gemv_wait(unsigned long long timeout_ns, cudaStream_t st) {
    unsigned int* err = nullptr;
    const cq_status se = device_error_word(&err);
    if (se != CQ_OK) return se;
    bounded_wait_probe_kernel<<<1, 32, 0, st>>>(err, timeout_ns);
    return check_launch();
}

unsigned int* gemv_error_word(int dev) {
    if (dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(g_err_mu);
    return g_gemv_err_ptr[dev];
}

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
    if (g != kGroup || K % kGroup != 0 || !cq_code_valid(b)) return CQ_ERR_INVALID_ARG;
    if (K > (1 << 24) || N > kMaxGemvRows || B > (1 << 30)) return CQ_ERR_UNSUPPORTED;
    if (!aligned16(packed) || !aligned16(norms) || !aligned16(Xq) || !aligned16(scale) ||
        !aligned16(Y))
        return CQ_ERR_ALIGNMENT;
    if (!workspace || workspace_bytes < cq_gemv_workspace_bytes(B, K)) return CQ_ERR_WORKSPACE;
    if (!aligned16(workspace)) return CQ_ERR_ALIGNMENT;
    if (K > 2 * kWarps2 * kSeg) return CQ_ERR_UNSUPPORTED;   // at most 2 segments per warp
    cudaStream_t st = as_stream(stream);
    // batches go through the tensor cores: the weights are read and decoded once for all
    // tokens (the workspace, B * K * 4 bytes, holds the fp16 activations)
    if (B >= kTensorMinBatch && N % 16 == 0)
        return gemv_tensor(packed, norms, N, K, b, cbk, Xq, scale, B, Y, workspace, st);
    // one or two tokens of 4-bit rows: 16-bit integer codewords (half the shared-memory
    // bytes per lookup), for at least 16 rows (fewer rows keep the fp32 codewords: one
    // small output of a short vector would magnify the codeword rounding)
    if (b == 4 && B <= 2 && N >= 16 && K % 1024 == 0) {
        const cq_status s = cq4_gemv_fx(packed, norms, N, K, cbk, Xq, scale, B, Y, st);
        if (s != CQ_ERR_UNSUPPORTED) return s;
    }
    // one token of 1-bit, 2-bit or ternary rows: the table-lookup kernel (one lookup and
    // one add per 4-bit nibble, lut.cu) once every SM gets a full block of 16 rows; its
    // per-CTA table costs more than it saves on fewer rows
    if ((b == 1 || b == 2 || b == CQ_TERNARY) && B == 1 && N >= 16 * (int64_t)sm_count())
        return cq_gemv_lut(packed, norms, N, K, g, b, cbk, Xq, scale, B, Y, stream);
    // segments per warp: 1 up to 16 segments (K <= 16384), else 2 (K <= 32768); two
    // tokens per pass when each warp owns a single segment
    const int nseg = (int)((K + kSeg - 1) / kSeg);
    const int spw = (nseg + kWarps2 - 1) / kWarps2;
    const int tb = (spw == 1 && B > 1) ? 2 : 1;
    // a single pass rotates the activations in its prologue; several passes share one
    // rotation kernel's output in the workspace
    const bool fused = B <= tb;
    const int f = cq_field_bits(b);
    float* xr = reinterpret_cast<float*>(workspace);
    if (!fused) {
        const int64_t groups = B * (K / kGroup);
        int64_t grid = (groups + 7) / 8;
        const int64_t cap = (int64_t)sm_count() * 16;
        if (grid > cap) grid = cap;
        const cq_status s = launch_pdl(rotate_act_kernel, dim3((unsigned)grid), dim3(kThreads), 0, st, Xq,
                                       groups, xr);
        if (s != CQ_OK) return s;
    }
    CqGemvParams p;
    {
        unsigned int* err = nullptr;
        const cq_status se = device_error_word(&err);
        if (se != CQ_OK) return se;
        p.err = err;
    }
    p.packed = packed; p.norms = norms; p.scale = scale; p.Y = Y;
    p.xr = fused ? nullptr : xr;
    p.xq = fused ? Xq : nullptr;
    p.N = N; p.K = (int)K; p.nseg = nseg;
    {
        // packed rows as 32-bit words (rows are 16 b-byte groups long, so 16-byte strides)
        const uint64_t rowbytes = (uint64_t)(K / kGroup) * 16u * (uint64_t)f;
        cq_status se = encode_map(&p.pmap, CU_TENSOR_MAP_DATA_TYPE_UINT32, packed, rowbytes / 4,
                                  (uint64_t)N, rowbytes, 32u * (uint32_t)f, kUnitRows);
        if (se != CQ_OK) return se;
        if (K % kSeg == 0) {   // norm rows of 8-group segments: 16-byte strides and boxes
            se = encode_map(&p.nmap, CU_TENSOR_MAP_DATA_TYPE_UINT16, norms, (uint64_t)(K / kGroup),
                            (uint64_t)N, (uint64_t)(K / kGroup) * 2u, 8u, kUnitRows);
            if (se != CQ_OK) return se;
        }
    }
    cq_host_levels(p.lv, b, cbk);
    p.rg = row_groups(p.nseg);
    for (int64_t t0 = 0; t0 < B; t0 += tb) {
        p.t0 = (int)t0;
        p.ntok = (int)((B - t0) < tb ? (B - t0) : tb);
        cq_status s;
        switch (f) {   // the ternary code runs the 2-bit kernel on its own level table
            case 1: s = dispatch_cq<1>(p, tb, spw, st); break;
            case 2: s = dispatch_cq<2>(p, tb, spw, st); break;
            case 3: s = dispatch_cq<3>(p, tb, spw, st); break;
            default: s = dispatch_cq<4>(p, tb, spw, st); break;
        }
        if (s != CQ_OK) return s;
    }
    return CQ_OK;
}

extern "C" cq_status q4_0_gemv(const uint8_t* blocks, int64_t N, int64_t K, const float* X,
                               int64_t B, float* Y, void* stream) {
    if (!blocks || !X || !Y || N < 1 || K < 1 || B < 1) return CQ_ERR_INVALID_ARG;
    if (K > 2 * kWarps2 * kSeg || N > kMaxGemvRows || B > (1 << 30)) return CQ_ERR_UNSUPPORTED;
    if (!aligned16(blocks) || !aligned16(X) || !aligned16(Y)) return CQ_ERR_ALIGNMENT;
    Q40GemvParams p;
    p.blocks = blocks; p.X = X; p.Y = Y; p.N = N; p.K = (int)K;
    p.nblk = (int)((K + 31) / 32);
    p.nseg = (p.nblk + 31) / 32;
    p.total_bytes = N * (int64_t)p.nblk * 18;
    cudaStream_t st = as_stream(stream);
    unsigned int* err = nullptr;
    {
        const cq_status se = device_error_word(&err);
        if (se != CQ_OK) return se;
    }
    p.err = err;
    // ring staging by tensor copies needs 16-byte row strides: 8 | nblk
    const bool bulk = (p.nblk % 8) == 0;
    if (bulk) {
        const uint64_t rowbytes = (uint64_t)p.nblk * 18u;
        const cq_status se = encode_map(&p.bmap, CU_TENSOR_MAP_DATA_TYPE_UINT32, blocks, rowbytes / 4,
                                        (uint64_t)N, rowbytes, kQSeg / 4, kUnitRows);
        if (se != CQ_OK) return se;
    }
    const int spw = (p.nseg + kWarps2 - 1) / kWarps2;
    p.rg = row_groups(p.nseg);
    const int tb = (spw == 1 && B > 1) ? 2 : 1;
    for (int64_t t0 = 0; t0 < B; t0 += tb) {
        p.t0 = (int)t0;
        p.ntok = (int)((B - t0) < tb ? (B - t0) : tb);
        cq_status s;
        if (bulk) {
            s = (spw == 2) ? run_q4_0_gemv<1, 2, true>(p, st)
              : (tb == 2) ? run_q4_0_gemv<2, 1, true>(p, st) : run_q4_0_gemv<1, 1, true>(p, st);
        } else {
            s = (spw == 2) ? run_q4_0_gemv<1, 2, false>(p, st)
              : (tb == 2) ? run_q4_0_gemv<2, 1, false>(p, st) : run_q4_0_gemv<1, 1, false>(p, st);
        }
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
    if (g != kGroup || K % kGroup != 0 || !cq_code_valid(b)) return CQ_ERR_INVALID_ARG;
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
