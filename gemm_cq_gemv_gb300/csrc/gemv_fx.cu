// CQ GEMV for 4-bit indices on 16-bit integer codewords (A4 + A5 at batch 1 and 2).
//
// The product of one row with one token is ("14MB 装下 45M 参数…", §一 and §三, with the
// rotation identity dot(w_g, x_g) = (norm / 128) * dot(cb[idx], Hu x_g)):
//
//   y[t][o] = s_t / 128 * sum_j norm[o][j] * sum_i cb[idx[o][j][i]] * xr[t][128 j + i]
//
// where xr = Hu q is the rotated int8 activation, an integer with |xr| <= 128 * 127.
//
// What sets the pace on the CUDA cores is the lookup of the codewords, not the bytes: a
// pair of fp32 codewords per lookup moves 4 bytes of shared memory per weight, which at
// 128 bytes per clock per SM caps a batch-1 4-bit GEMV near 0.62 of the GB300's copy
// bandwidth.  Here a lookup moves 2 bytes per weight and the sums are exact integers:
//
//   * the codewords enter as 16-bit fixed-point integers C = rint(cb * S), S =
//     floor(32767 / max |cb|);
//   * a shared table holds, for every byte of packed indices (a pair of 4-bit indices
//     a = low nibble, b = high nibble), the word [lo(C_a), lo(C_b), hi(C_a), hi(C_b)]
//     (lo the unsigned low byte, hi the signed high byte, C = 256 hi + lo), one copy per
//     lane so that every lookup is free of bank conflicts;
//   * the activations sit in registers as pairs (xr_a, xr_b) of int16;
//   * dp2a.lo adds xr_a lo(C_a) + xr_b lo(C_b) and dp2a.hi adds xr_a hi(C_a) + xr_b hi(C_b);
//   * a lane's 32 positions lie inside one 128-group, so its sum 256 H + L is scaled once
//     by the group's fp16 norm and accumulated in fp32.
//
// The only departure from fp32 codewords is the rounding of each codeword to the 16-bit
// grid, at most 0.5 / S (<= 4.2e-5 for the Lloyd-Max tables), well inside the 1e-3
// bound of the product; the host sends rows fewer than 16 (where one small output could
// magnify it) to the fp32-codeword kernel.
//
// Layout of the work: one CTA of NW warps per SM (32 for one token, 16 for two, whose
// activations take twice the registers), persistent over groups of 8 rows.  Warp w owns
// the K-segment (w mod nsl) of 1024 positions - lane l the positions [32 l, 32 l + 32) -
// and belongs to warp set w / nsl; the nsl warps of a set share each of its row groups.
// Row group j goes to CTA j mod G and, in turn, to the CTA's warp sets, so every CTA
// holds the same number of groups (+-1) and a set that finishes early leaves the SM's
// issue slots to the others.  Packed rows arrive through a per-warp ring of kFxRing slots
// of 2 rows x one segment (1 KB), each filled by one tensor copy issued by one lane; a
// warp starts its first copies as soon as its own ring barriers exist, before the table
// is built and the activations are rotated.  The tensor-copy unit starts at most ~47
// copies per microsecond per SM (measured), so the copies are whole units and nothing
// else: the group norms of a row group (8 rows x 8 groups of a segment, 128 bytes) come
// with one 4-byte load per lane, issued a group ahead, and reach the lanes that need them
// by warp shuffles.  The partial sums of a row group are added across its set's warps in
// warp order (deterministic).  When several warp sets share a segment (K <= 8192), each
// 128-group of activations is rotated once, by one warp, and shared in shared memory.

#include <mutex>

#include "gemv_pipe.cuh"

namespace cq {
namespace {

using namespace pipe;

constexpr int kFxSeg = 1024;                 // positions per warp segment
constexpr int kFxUnitRows = 2;               // rows per staged unit
constexpr int kFxRing = 4;                   // slots per warp ring (slot = unit & 3)
constexpr uint32_t kFxSegBytes = 512;        // a 4-bit row segment
constexpr uint32_t kFxSlot = kFxUnitRows * kFxSegBytes;   // packed rows of one unit (1 KB)
constexpr uint32_t kFxTable = 65536;         // 256 entries x 256-byte stride (lanes use 128)
constexpr size_t kFxSmem = 227 * 1024;
static_assert(kFxRing == 4, "slot and phase arithmetic assume 4 slots");
static_assert(kRows % kFxUnitRows == 0, "a tile is a whole number of units");
// The lanes' copies of a table entry fill the first 128 bytes of its 256-byte stride; the
// other 128 bytes of the 256 entries ("holes", 128-byte aligned) hold the partial sums of
// the cross-warp reduction (holes 128 .. 255, four 8-float partials each).
__host__ __device__ constexpr uint32_t hole(uint32_t i) { return i * 256u + 128u; }
constexpr uint32_t kFxPartHole = 128;
template <int NW, int TB>
constexpr bool holes_fit() { return kSlots * NW * TB <= 4 * 128; }

struct Cq4FxParams {
    CUtensorMap pmap;        // packed rows as [N][K / 8] uint32, box 128 x kFxUnitRows
    const uint16_t* norms;   // [N][K / 128] fp16
    const int8_t* xq;        // [B][K] int8 activations, rotated in the prologue
    const float* scale;      // [B]
    float* Y;                // [B][N]
    unsigned int* err;       // device error word
    int64_t N;
    int K;
    int nseg;                // K / 1024
    int rg;                  // row groups per tile
    int t0;                  // first token of this pass
    int ntok;                // tokens in this pass (<= TB)
    uint32_t smem_bytes;     // dynamic shared memory of the launch
    int share;               // 1: each 128-group rotated once per CTA, shared in shared memory
    int64_t groups_base;     // a CTA takes groups_base row groups (8 rows), one more if
    int groups_extra;        //   blockIdx.x < groups_extra
    float out_scale;         // 1 / (128 S)
    int cw[16];              // the 16-bit codewords C_t
};

// shared address of (pair entry = byte J of wv, this lane): base | byte << 8 | lane << 2
template <int J>
__device__ __forceinline__ uint32_t entry_addr(uint32_t wv, uint32_t lb) {
    uint32_t a;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(a) : "r"(wv), "r"(lb), "n"(0x7604 | (J << 4)));
    return a;
}
__device__ __forceinline__ int dp2a_lo(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp2a.lo.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ int dp2a_hi(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp2a.hi.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ uint32_t lds_u32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}

// xr = Hu q for this lane's 32 positions of a 128-group held by lanes 4g..4g+3, in
// integers: five butterfly stages inside the lane, the strides of 32 and 64 across lanes
__device__ __forceinline__ void rotate32_int(int (&v)[32], int lane) {
#pragma unroll
    for (int h = 1; h < 32; h <<= 1)
#pragma unroll
        for (int j = 0; j < 32; ++j)
            if ((j & h) == 0) {
                const int a = v[j], b = v[j + h];
                v[j] = a + b;
                v[j + h] = a - b;
            }
#pragma unroll
    for (int m = 1; m <= 2; m <<= 1) {
        const bool upper = (lane & m) != 0;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const int q = __shfl_xor_sync(0xffffffffu, v[j], m);
            v[j] = upper ? (q - v[j]) : (v[j] + q);
        }
    }
}

// xr = Hu q of one 128-group held by a warp, lane l with positions 4l..4l+3: spans 1 and 2
// inside the lane, 4..64 across lanes (exact integers)
__device__ __forceinline__ void rotate128_int(int (&v)[4], int lane) {
    const int a0 = v[0] + v[1], a1 = v[0] - v[1], a2 = v[2] + v[3], a3 = v[2] - v[3];
    v[0] = a0 + a2; v[2] = a0 - a2; v[1] = a1 + a3; v[3] = a1 - a3;
#pragma unroll
    for (int m = 1; m <= 16; m <<= 1) {
        const bool upper = (lane & m) != 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int q = __shfl_xor_sync(0xffffffffu, v[j], m);
            v[j] = upper ? (q - v[j]) : (v[j] + q);
        }
    }
}

template <int NW, int TB>
__global__ void __launch_bounds__(NW * 32, 1) cq4_gemv_fx_kernel(const __grid_constant__ Cq4FxParams p) {
    extern __shared__ __align__(128) unsigned char smem_f[];
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    pdl_trigger();
    // shared plan: the table in a 64 KB aligned window (its address is one byte permute),
    // everything else first-fit in the space below and above it
    const uint32_t sbase = smem_u32(smem_f), send = sbase + p.smem_bytes;
    const uint32_t tbase = (sbase + 65535u) & ~65535u;
    SmemCarve cv;
    cv.ok = tbase + kFxTable <= send;
    cv.a = sbase; cv.a_end = tbase; cv.b = tbase + kFxTable; cv.b_end = send;
    static_assert(holes_fit<NW, TB>(), "the partials must fit the table's holes");
    const uint32_t red_at = cv.take((uint32_t)p.rg * kSlots * (8 + 4), 8);   // slot barriers, counters
    const uint32_t bar_at = cv.take(NW * kFxRing * 8, 8);
    // the NW rings (equal sizes: first-fit fills the space below the table, then above)
    uint32_t ring_at;
    {
        constexpr uint32_t kRingB = kFxRing * kFxSlot;
        const uint32_t a0 = (cv.a + 127u) & ~127u, b0 = (cv.b + 127u) & ~127u;
        const uint32_t na = a0 < cv.a_end ? (cv.a_end - a0) / kRingB : 0u;
        const uint32_t nb = (uint32_t)NW > na ? (uint32_t)NW - na : 0u;
        ring_at = (uint32_t)w < na ? a0 + (uint32_t)w * kRingB : b0 + ((uint32_t)w - na) * kRingB;
        if (na > 0u) cv.a = a0 + (na < (uint32_t)NW ? na : (uint32_t)NW) * kRingB;
        if (nb > 0u) {
            cv.b = b0 + nb * kRingB;
            if (cv.b > cv.b_end) cv.ok = false;
        }
    }
    const uint32_t xr_at = p.share ? cv.take((uint32_t)TB * (uint32_t)p.K * 2u, 16) : 0u;
    if (!cv.ok) {   // the launch's shared memory cannot hold the plan (host sizing error)
        if (tid == 0) atomicOr(p.err, 4u);
        return;
    }
    auto gen = [&](uint32_t a) { return smem_f + (a - sbase); };
    Reduce rd;
    rd.part = reinterpret_cast<float*>(gen(tbase + hole(kFxPartHole)));
    rd.pstride = 64;   // 256 bytes from one hole to the next
    rd.empty = reinterpret_cast<uint64_t*>(gen(red_at));
    rd.count = reinterpret_cast<uint32_t*>(rd.empty + p.rg * kSlots);
    uint64_t* rfull = reinterpret_cast<uint64_t*>(gen(bar_at)) + w * kFxRing;
    uint8_t* ring = gen(ring_at);
    if (tid == 0) prefetch_tensormap(&p.pmap);
    // a warp's ring barriers are its own: it initialises them and starts its first copies
    // at once; the table, the activations and the rotation overlap those copies
    if (lane < kFxRing) mbar_init(&rfull[lane], 1);
    for (int i = tid; i < p.rg * kSlots; i += NW * 32) {
        rd.count[i] = 0u;
        mbar_init(&rd.empty[i], 1);
    }
    if (lane == 0) asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    __syncwarp();

    const int nsl = p.nseg < NW ? p.nseg : NW;
    const int slot = w % nsl, rgi = w / nsl;
    const bool busy = rgi < p.rg;
    // row group j (rows 8 j .. 8 j + 7) belongs to CTA j mod G; the CTA's m-th group goes
    // to warp set m mod rg as that set's (m / rg)-th: every CTA holds the same number of
    // groups (+-1), and sets that finish early leave the SM's issue slots to the others
    const int64_t ncta = p.groups_base + ((int)blockIdx.x < p.groups_extra ? 1 : 0);
    const int64_t ngr = busy && ncta > rgi ? (ncta - rgi + p.rg - 1) / p.rg : 0;   // this set's groups
    const int64_t gstep = (int64_t)kRows * p.rg * gridDim.x;                        // rows between them
    const int64_t row0 = (int64_t)kRows * (blockIdx.x + (int64_t)rgi * gridDim.x);  // first row
    constexpr int upt = kRows / kFxUnitRows;                    // units per row group
    const int64_t U = ngr * upt;

    // cursor of the next unit to issue (units go out strictly in order)
    int64_t nx_base = row0;
    int nx_rem = 0;
    auto issue = [&](int d) {
        if (lane == 0) {
            const int y = (int)(nx_base + nx_rem * kFxUnitRows);
            mbar_arrive_tx(&rfull[d], kFxSlot);
            tma_box(ring + d * kFxSlot, &p.pmap, slot * (kFxSegBytes / 4), y, &rfull[d]);
        }
        if (++nx_rem == upt) {
            nx_rem = 0;
            nx_base += gstep;
        }
    };
    // The packed rows are read before the wait for the previous kernel of the stream:
    // weights come from kernels that release their dependents only at completion (the
    // library's encoders), so that wait concerns the activations alone, and the first
    // copies' latency overlaps the previous kernel's tail.
    if (busy)
        for (int64_t u = 0; u < kFxRing - 1 && u < U; ++u) issue((int)u);

    // pair table: entry e (a = e & 15, b = e >> 4) = [lo(C_a), lo(C_b), hi(C_a), hi(C_b)]
    // at tbase + e * 256 + lane * 4; a thread writes one entry's copies for eight lanes
    // (lane l holds C_(l & 15); 1024 is a multiple of the block, so every lane takes part)
    const int cwl = p.cw[lane & 15];
    for (int i = tid; i < 256 * 4; i += NW * 32) {
        const int e = i >> 2;
        const uint32_t ca = (uint32_t)__shfl_sync(0xffffffffu, cwl, e & 15);
        const uint32_t cb = (uint32_t)__shfl_sync(0xffffffffu, cwl, e >> 4);
        const uint32_t word = (ca & 0xFFu) | (cb & 0xFFu) << 8 | ((ca >> 8) & 0xFFu) << 16 | ((cb >> 8) & 0xFFu) << 24;
        const uint4 v4 = make_uint4(word, word, word, word);
        uint4* dst = reinterpret_cast<uint4*>(gen(tbase + (uint32_t)e * 256u + (uint32_t)(i & 3) * 32u));
        dst[0] = v4;
        dst[1] = v4;
    }
    pdl_wait();   // the activations may come from the previous kernel
    // this lane's activations: int8 -> Hu q (exact integers) -> int16 pairs
    uint32_t xp[TB][16];
    if (p.share) {
        // the segment's eight groups are rotated by its p.rg warps, one group at a time,
        // and land in shared memory as int16; each lane then reads its 32 positions
        int16_t* xs = reinterpret_cast<int16_t*>(gen(xr_at));
        if (busy) {
#pragma unroll
            for (int t = 0; t < TB; ++t) {
                for (int g = rgi; g < 8; g += p.rg) {
                    const int pos = slot * kFxSeg + g * kGroup + 4 * lane;
                    char4 c = make_char4(0, 0, 0, 0);
                    if (t < p.ntok) c = *reinterpret_cast<const char4*>(p.xq + (int64_t)(p.t0 + t) * p.K + pos);
                    int v[4] = {c.x, c.y, c.z, c.w};
                    rotate128_int(v, lane);
                    const uint2 pr = make_uint2(((uint32_t)v[0] & 0xFFFFu) | ((uint32_t)v[1] << 16),
                                                ((uint32_t)v[2] & 0xFFFFu) | ((uint32_t)v[3] << 16));
                    *reinterpret_cast<uint2*>(xs + (size_t)t * p.K + pos) = pr;
                }
            }
        }
        __syncthreads();   // table and rotated groups complete
#pragma unroll
        for (int t = 0; t < TB; ++t) {
            const uint4* src = reinterpret_cast<const uint4*>(xs + (size_t)t * p.K + slot * kFxSeg + lane * 32);
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                const uint4 q = src[h];
                xp[t][4 * h] = q.x; xp[t][4 * h + 1] = q.y; xp[t][4 * h + 2] = q.z; xp[t][4 * h + 3] = q.w;
            }
        }
    } else {
#pragma unroll
        for (int t = 0; t < TB; ++t) {
            const bool ok = busy && t < p.ntok;
            const int8_t* src = p.xq + (int64_t)(p.t0 + t) * p.K + slot * kFxSeg + lane * 32;
            int v[32];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int4 c = ok ? *reinterpret_cast<const int4*>(src + 16 * h) : make_int4(0, 0, 0, 0);
                const int wv[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
                for (int q = 0; q < 16; ++q) v[16 * h + q] = (int)(int8_t)(wv[q >> 2] >> (8 * (q & 3)));
            }
            rotate32_int(v, lane);
#pragma unroll
            for (int q = 0; q < 16; ++q)
                xp[t][q] = ((uint32_t)v[2 * q] & 0xFFFFu) | ((uint32_t)v[2 * q + 1] << 16);
        }
        __syncthreads();   // table complete
    }
    if (!busy) return;   // warps left over when the segments do not divide the CTA

    const uint32_t lb = tbase | ((uint32_t)lane << 2);
    const int grp = lane >> 2;   // this lane's group within a segment's 8
    // group norms of a tile: lane l holds the two of (row l / 4, groups 2 (l % 4) + 0, 1 of
    // the segment)
    const int G = p.K / kGroup;
    auto load_norms = [&](int64_t k) -> uint32_t {
        const int64_t row = row0 + k * gstep + (lane >> 2);
        if (k >= ngr || row >= p.N) return 0u;
        return __ldg(reinterpret_cast<const uint32_t*>(p.norms + row * G + slot * 8 + 2 * (lane & 3)));
    };
    uint32_t nrm_next = load_norms(0);
    int64_t u = 0;
    for (int64_t k = 0; k < ngr; ++k) {
        const int64_t rbase = row0 + k * gstep;   // the group's first row
        const uint32_t nrm_tile = nrm_next;
        nrm_next = load_norms(k + 1);   // a group ahead
        float acc[TB][kRows];
#pragma unroll
        for (int t = 0; t < TB; ++t)
#pragma unroll
            for (int r = 0; r < kRows; ++r) acc[t][r] = 0.0f;
#pragma unroll
        for (int h = 0; h < upt; ++h, ++u) {
            if (u + kFxRing - 1 < U) {
                __syncwarp();   // every lane is done with the slot about to be refilled
                if (lane == 0) fence_proxy_async();
                issue((int)((u + kFxRing - 1) & (kFxRing - 1)));
            }
            const int d = (int)(u & (kFxRing - 1));
            const uint8_t* sp = ring + d * kFxSlot;
            mbar_wait(&rfull[d], (uint32_t)(u >> 2) & 1u, p.err);
#pragma unroll
            for (int r = 0; r < kFxUnitRows; ++r) {
                const uint4 wq = *reinterpret_cast<const uint4*>(sp + r * kFxSegBytes + lane * 16);
                const uint32_t wd[4] = {wq.x, wq.y, wq.z, wq.w};
                int lo[TB][2], hi[TB][2];
#pragma unroll
                for (int t = 0; t < TB; ++t) lo[t][0] = lo[t][1] = hi[t][0] = hi[t][1] = 0;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint32_t c0 = lds_u32(entry_addr<0>(wd[kk], lb));
                    const uint32_t c1 = lds_u32(entry_addr<1>(wd[kk], lb));
                    const uint32_t c2 = lds_u32(entry_addr<2>(wd[kk], lb));
                    const uint32_t c3 = lds_u32(entry_addr<3>(wd[kk], lb));
#pragma unroll
                    for (int t = 0; t < TB; ++t) {
                        lo[t][0] = dp2a_lo(xp[t][4 * kk + 0], c0, lo[t][0]);
                        hi[t][0] = dp2a_hi(xp[t][4 * kk + 0], c0, hi[t][0]);
                        lo[t][1] = dp2a_lo(xp[t][4 * kk + 1], c1, lo[t][1]);
                        hi[t][1] = dp2a_hi(xp[t][4 * kk + 1], c1, hi[t][1]);
                        lo[t][0] = dp2a_lo(xp[t][4 * kk + 2], c2, lo[t][0]);
                        hi[t][0] = dp2a_hi(xp[t][4 * kk + 2], c2, hi[t][0]);
                        lo[t][1] = dp2a_lo(xp[t][4 * kk + 3], c3, lo[t][1]);
                        hi[t][1] = dp2a_hi(xp[t][4 * kk + 3], c3, hi[t][1]);
                    }
                }
                const int row = h * kFxUnitRows + r;
                const uint32_t nv = __shfl_sync(0xffffffffu, nrm_tile, row * 4 + (grp >> 1));
                const float nrm = f16_bits_to_f32((uint16_t)((grp & 1) ? (nv >> 16) : nv));
#pragma unroll
                for (int t = 0; t < TB; ++t) {
                    // |lo| <= 32 * 16256 * 255 and |hi| <= 32 * 16256 * 128: no int32 overflow
                    const float v = fmaf((float)(hi[t][0] + hi[t][1]), 256.0f, (float)(lo[t][0] + lo[t][1]));
                    acc[t][row] = fmaf(nrm, v, acc[t][row]);
                }
            }
        }
        group_reduce<TB, NW>(rd, acc, (int)k, w, lane, nsl, rgi, p.ntok, p.err,
                             [&](int t, int r, float sum) {
                                 const int64_t row = rbase + r;
                                 if (row < p.N) {
                                     const int tok = p.t0 + t;
                                     p.Y[(int64_t)tok * p.N + row] = sum * (p.scale[tok] * p.out_scale);
                                 }
                             });
    }
}

template <int NW, int TB>
cq_status run_cq4_fx(Cq4FxParams p, cudaStream_t st) {
    static bool attr[64] = {};
    static std::mutex mu;
    auto kern = cq4_gemv_fx_kernel<NW, TB>;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return check_launch();
    if (dev < 0 || dev >= 64) return CQ_ERR_UNSUPPORTED;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!attr[dev]) {
            if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kFxSmem) !=
                cudaSuccess)
                return check_launch();
            attr[dev] = true;
        }
    }
    p.smem_bytes = (uint32_t)kFxSmem;
    const int64_t ngroups = (p.N + kRows - 1) / kRows;
    int64_t grid = sm_count();
    if (ngroups < grid) grid = ngroups;
    p.groups_base = ngroups / grid;
    p.groups_extra = (int)(ngroups % grid);
    // several warps per segment: rotate each group once and share it (TB * K * 2 bytes of
    // shared memory beside the rings and the table)
    p.share = (p.rg >= 2 && p.K <= 8192) ? 1 : 0;
    return launch_pdl(kern, dim3((unsigned)grid), dim3(NW * 32), kFxSmem, st, p);
}

}  // namespace

// The 16-bit codeword grid of the 4-bit kernel: S = floor(32767 / max |cb|) and
// C_t = rint(cb_t * S); false when the levels are not all finite or all zero (the
// fp32-codeword kernel then runs).
bool cq4_fx_codewords(const float (&lv)[16], int (&cw)[16], float* out_scale) {
    double amax = 0.0;
    for (int t = 0; t < 16; ++t) {
        const double a = lv[t] < 0 ? -(double)lv[t] : (double)lv[t];
        if (!(a <= 3.0e38)) return false;   // inf or nan
        if (a > amax) amax = a;
    }
    if (!(amax > 1.0e-30)) return false;
    double S = __builtin_floor(32767.0 / amax);
    if (S < 1.0) S = 1.0;
    for (int t = 0; t < 16; ++t) {
        const double c = __builtin_rint((double)lv[t] * S);
        cw[t] = (int)(c > 32767.0 ? 32767.0 : (c < -32767.0 ? -32767.0 : c));
    }
    *out_scale = (float)(1.0 / (128.0 * S));
    return true;
}

// Batch-1 and batch-2 CQ GEMV of 4-bit rows on 16-bit integer codewords.  Requires
// K % 1024 == 0, K <= 32768, 16-byte aligned operands (checked by the caller).
cq_status cq4_gemv_fx(const uint8_t* packed, const uint16_t* norms, int64_t N, int64_t K,
                      const cq_codebook* cbk, const int8_t* Xq, const float* scale, int64_t B,
                      float* Y, cudaStream_t st) {
    Cq4FxParams p;
    float lv[16];
    cq_host_levels(lv, 4, cbk);
    if (!cq4_fx_codewords(lv, p.cw, &p.out_scale)) return CQ_ERR_UNSUPPORTED;
    {
        unsigned int* err = nullptr;
        const cq_status se = device_error_word(&err);
        if (se != CQ_OK) return se;
        p.err = err;
    }
    p.norms = norms; p.xq = Xq; p.scale = scale; p.Y = Y;
    p.N = N; p.K = (int)K; p.nseg = (int)(K / kFxSeg);
    {
        const uint64_t rowbytes = (uint64_t)K / 2u;
        const cq_status se = encode_map(&p.pmap, CU_TENSOR_MAP_DATA_TYPE_UINT32, packed, rowbytes / 4,
                                        (uint64_t)N, rowbytes, kFxSegBytes / 4, kFxUnitRows);
        if (se != CQ_OK) return se;
    }
    // two tokens share a pass of the 16-warp kernel when each warp owns one segment
    // (K <= 16384); otherwise every token is a pass of the 32-warp kernel
    const int step = (B >= 2 && p.nseg <= 16) ? 2 : 1;
    for (int64_t t0 = 0; t0 < B; t0 += step) {
        p.t0 = (int)t0;
        p.ntok = (int)((B - t0) < step ? (B - t0) : step);
        cq_status s;
        if (p.ntok == 2) {
            p.rg = p.nseg >= 16 ? 1 : 16 / p.nseg;
            s = run_cq4_fx<16, 2>(p, st);
        } else {
            p.rg = p.nseg >= 32 ? 1 : 32 / p.nseg;
            s = run_cq4_fx<32, 1>(p, st);
        }
        if (s != CQ_OK) return s;
    }
    return CQ_OK;
}

}  // namespace cq
