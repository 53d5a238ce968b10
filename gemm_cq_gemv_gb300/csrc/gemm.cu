// Prefill GEMM for CQ-W4A8 weights on the 5th-generation tensor cores (A6).
//
// "14MB 装下 45M 参数…", §三: prefill is a GEMM over the same pre-transposed [out, in]
// rows the decode GEMV streams; §一: w_group = (cb[idx] * norm / sqrt(128)) @ H.  With
// xr = Hu @ q (the rotated int8 activations, exact integers) the product is
//   Y[t][o] = s_t / 128 * sum_k xr[t][k] * cb[idx[o][k]] * norm[o][k / 128]
// and both factors of the contraction are fed to tcgen05.mma as fp16:
//   A = fp16(fp16(cb[idx]) * norm)  [N out-rows][K]  - dequantised into TENSOR memory
//   B = fp16(xr * s_t / 128)        [M tokens][K]    - rotated once per call, TMA-loaded
// D[o][t] accumulates in fp32 in tensor memory; the epilogue rounds to bf16 and stores
// the transposed tile.  Keeping the dequantised weights in tensor memory means shared
// memory only carries the activation tile (TMA write + one MMA read) and the packed
// nibbles, which is what lets the MMA rate approach the tensor-core peak.
//
// One CTA per SM (persistent), tile = 128 out-rows x 192 tokens, K in chunks of 64.
// Shared memory: the codeword-pair table (64 KB, one copy per lane) at a 64 KB boundary of
// the shared window, so a lookup address is one byte permute; four 28 KB stages around it.
// Tensor memory (512 columns): 4 A stages of 32 columns (64 bf16 per row) and two
// 192-column fp32 accumulators (the epilogue of a tile overlaps the next main loop).
// Warp roles (prefill):
//   warp 0      TMA producer: per stage the activation tile (128-byte
//               swizzle) and the packed 4-bit weight tile (128 rows x 32 bytes)
//   warp 1      MMA issuer (one thread): 4 tcgen05.mma (M=128, N=192, K=16) per stage,
//               A from tensor memory, B from shared memory
//   warps 2-9   epilogue: tcgen05.ld (two warps per TMEM lane quarter, 96 tokens each,
//               16-column pieces),
//               bf16, store
//   warps 10-25 dequant, two groups of eight taking alternate stages (a stage's
//               dequant latency - table loads, tensor-memory store and its wait - is
//               longer than its share of the MMA time, so each group gets two stage
//               times per stage): packed tile -> fp16 codeword pairs from a per-lane
//               shared table, times the group norm, tcgen05.st into the A stage
//               (two warps per lane quarter, 32 k each)
// What paces the prefill, measured with clock stamps of CTA 0: the MMA issuer thread.
// Its wait, fence, four MMAs and commit take ~600-750 cycles per stage against ~490
// cycles of tensor work; each tcgen05 instruction costs the issuing thread ~60-90 cycles.
// The 32-token decode tiles run two copy threads (warp 0: activation tiles, warp 1:
// packed tiles or weight slabs) and MMAW issuer threads instead of one: the
// thread that issues a stage also waits for it, fences and commits it, and those steps
// (not the tensor core: an M=128, N=32 MMA is ~25 cycles of work) set the pace of one
// issuer, ~600 cycles per stage.  Issuer j takes the stages t of a tile with
// t % MMAW == j into a partial accumulator of its own; each tracks only its own MMAs
// with its commits, and the epilogue adds the partials.  The epilogue and dequant warps
// follow the copy and issuer warps.
// Every mbarrier wait is bounded (globaltimer); on expiry the CTA raises a device error
// flag, stops issuing work, frees its tensor memory and returns.

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <mutex>

#include "common.cuh"

namespace cq {
namespace {

constexpr int kBO = 128;                 // out-rows per tile (MMA M, TMEM lanes)
constexpr int kBK = 64;                  // K per stage (128 bytes of 16-bit operands)
constexpr int kEpiWarps = 8;             // two per TMEM lane quarter
constexpr int kDequantWarps = 8;         // per stage: two per TMEM lane quarter
constexpr int kDequantGroups = 2;        // the first eight dequant warps take even stages
constexpr int kTmemCols = 512;
constexpr int kACols = kBK / 2;                       // 32 TMEM columns per A stage
constexpr int kGemmSmem = 227 * 1024;    // table (64 KB, 64 KB aligned) + stages + barriers
constexpr int kBarBytes = 512;           // barrier block: barriers, TMEM slot, flags, levels
constexpr int kMaxProblems = 120;
constexpr int kMaxCtaTiles = 256;        // tiles per CTA whose lookup is precomputed in shared memory
constexpr int kMaxActs = 8;

// Q4_0 weights reach shared memory in slabs of 256 k (8 blocks, 144 bytes per row: the
// smallest 16-byte multiple of the 18-byte block), on a ring of slabs; each slab feeds
// four 64-k stages.  1- and 3-bit CQ rows (8 and 24 bytes per 64-k stage, no legal
// tensor-copy box) take the same ring with slabs of two stages (16 and 48 bytes per row).
constexpr int kQSlabRowBytes = 144;

enum WeightFormat { kFmtCQ = 0, kFmtQ40 = 1 };

// Tile configuration of one kernel instance.
//   BT      tokens per tile (MMA N)
//   F16     fp16 operands and fp32 output (the batched-decode form of the product);
//           otherwise bf16 operands and bf16 output (prefill)
//   STAGES  depth of the shared-memory ring (= tensor-memory A stages)
//   FMT     weight format: CQ (packed indices + norms) or Q4_0 blocks
//   SLABS   Q4_0 and 1-/3-bit CQ: depth of the weight-slab ring
//   TLIST   look the CTA's tiles up once, into shared memory (grouped launches of many
//           problems, where each lookup is a binary search over the parameter block)
//   BITS    CQ index width: 4 or 2 (the packed tile rides in the stage, 32 or 16 bytes
//           per row), 1 or 3 (slabs of two stages)
//   PF16    fp16 codeword pairs and fp16 operands with bf16 output (prefill)
//   MMAW    MMA issuer threads, each with a partial accumulator per buffer
//   PROD    copy-issuing threads: 1, or 2 (one for the activation tiles, one for the
//           packed weight tiles or slabs)
template <int BT_, bool F16_, int STAGES_, int FMT_ = kFmtCQ, int SLABS_ = 0, bool TLIST_ = false,
          int BITS_ = 4, bool PF16_ = false, int MMAW_ = 1, int PROD_ = 1>
struct GemmCfg {
    static constexpr int BT = BT_;
    static constexpr bool F16 = F16_;
    // PF16: fp16 operands with the bf16 output of the prefill; the dequant looks up fp16
    // codeword pairs and scales them by the fp16 norm with one multiply
    static constexpr bool PF16 = PF16_;
    static constexpr bool OPF16 = F16 || PF16;     // fp16 (not bf16) MMA operands
    static constexpr int BITS = BITS_;
    static constexpr bool CQSLAB = FMT_ == kFmtCQ && (BITS == 1 || BITS == 3);
    // fp16 codeword pairs scaled by the fp16 norm with one multiply: every CQ tile with
    // fp16 operands whose packed indices ride in the stage (4 and 2 bits)
    static constexpr bool HPAIR = FMT_ == kFmtCQ && !CQSLAB && OPF16;
    static constexpr int STAGES = STAGES_;
    static constexpr int FMT = FMT_;
    static constexpr int SLABS = SLABS_;
    static constexpr bool TLIST = TLIST_;
    static constexpr int PTILE = FMT == kFmtCQ && !CQSLAB ? kBO * kBK * BITS / 8 : 0;   // packed bytes per stage
    static constexpr int SPS = FMT == kFmtQ40 ? 4 : 2;                            // stages per slab
    static constexpr int SLABROW = FMT == kFmtQ40 ? kQSlabRowBytes : SPS * kBK * BITS / 8;
    static constexpr int SLABBYTES = kBO * SLABROW;
    static constexpr int XTILE = BT * kBK * 2;        // activation tile bytes
    static constexpr int STAGE = XTILE + PTILE;
    static constexpr int DCOL0 = STAGES * kACols;     // accumulators after the A stages
    static constexpr int MMAW = MMAW_;
    static constexpr int PROD = PROD_;
    static constexpr int EPI0 = PROD + MMAW;           // first epilogue warp
    static constexpr int DEQ0 = EPI0 + kEpiWarps;      // first dequant warp
    static constexpr int THREADS = (DEQ0 + kDequantGroups * kDequantWarps) * 32;
    static_assert((BT / (kEpiWarps / 4)) % 16 == 0, "epilogue warps: 16-column pieces");
    static_assert(THREADS <= 1024, "one CTA per SM");
    static_assert(PROD == 1 || PROD == 2, "one or two copy-issuing threads");
    static_assert(DCOL0 + 2 * MMAW * BT <= kTmemCols, "tensor memory budget");
    static_assert(MMAW == 1 || BT == 32, "several issuers: 32-token tiles");
    static_assert(STAGE % 1024 == 0, "stages keep the 1024-byte swizzle alignment");
    static_assert((3 * STAGES + 4 + 2 * SLABS) * 8 + 16 + 64 <= kBarBytes, "barrier block");
    static_assert(FMT == kFmtCQ || (F16 && SLABS >= 2), "Q4_0 runs with fp16 operands on a slab ring");
    static_assert(BITS == 4 || (FMT == kFmtCQ && F16), "1- to 3-bit CQ rows: decode batches only");
    static_assert(!CQSLAB || SLABS >= 2, "1- and 3-bit CQ rows run on a slab ring");
    static_assert(FMT == kFmtQ40 || CQSLAB || SLABS == 0, "4- and 2-bit CQ tiles ride in the stages");
    static_assert(!PF16 || (!F16 && FMT == kFmtCQ && BITS == 4), "fp16 pair tables: 4-bit prefill");
};
using PrefillCfg = GemmCfg<192, false, 4, kFmtCQ, 0, true, 4, true>;   // 24 KB activation tile, 28 KB stages
constexpr int kDecodeIssuers = 2;
constexpr int kDecodeProducers = 2;
using DecodeCfg = GemmCfg<32, true, 8, kFmtCQ, 0, false, 4, false, kDecodeIssuers, kDecodeProducers>;   // 4 KB activation tile, 8 KB stages
using Decode2Cfg = GemmCfg<32, true, 8, kFmtCQ, 0, false, 2, false, kDecodeIssuers, kDecodeProducers>;  // 2-bit rows: 6 KB stages
using Decode1Cfg = GemmCfg<32, true, 8, kFmtCQ, 4, false, 1, false, kDecodeIssuers, kDecodeProducers>;  // 1-bit rows: 4 KB stages + 2 KB slabs
using Decode3Cfg = GemmCfg<32, true, 8, kFmtCQ, 4, false, 3, false, kDecodeIssuers, kDecodeProducers>;  // 3-bit rows: 4 KB stages + 6 KB slabs
using Q40WideCfg = GemmCfg<192, true, 4, kFmtQ40, 4>;    // Q4_0, many tokens: 96 + 72 KB
using Q40NarrowCfg = GemmCfg<32, true, 8, kFmtQ40, 4, false, 4, false, kDecodeIssuers, kDecodeProducers>;   // Q4_0, up to 32 tokens: 32 + 72 KB

struct GemmProblem {
    CUtensorMap pmap;        // packed bytes as [N][K/2] uint8, box 32 x 128
    const uint8_t* packed;   // [N][K/128][64]
    const uint16_t* norms;   // [N][K/128]
    const float* scale;      // [M]
    void* Y;                 // [M][N] bf16 (prefill) or fp32 (decode)
    int N, K;
    int act;                 // index of the activation tensor map
    int tiles_n;
    int tile_begin;          // first global tile index of this problem
    int tiles_per_split;     // tiles_n * tiles_m
    int ksplit;              // 1, or 2: each output tile is two half-K tiles whose fp32
                             // partials are added into Y (zeroed by the host)
    int kchunk;              // stages of one split
};

struct GemmParams {
    CUtensorMap tmap[kMaxActs];
    GemmProblem prob[kMaxProblems];
    int nprob;
    int M;
    int tiles_m;
    int total_tiles;
    float lv[16];
    unsigned int* err;
    unsigned long long timeout_ns;
};

// ---- small PTX wrappers -----------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(b)), "r"(count));
}
__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(b))
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive_tx(uint64_t* b, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                     smem_u32(b)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try(uint64_t* b, uint32_t parity) {
    uint32_t ok;
    // with a suspend-time hint the waiting thread sleeps until the phase completes (or
    // the hint elapses) instead of spinning and taking issue slots from working warps
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(smem_u32(b)), "r"(parity), "r"(1000000u)
        : "memory");
    return ok != 0;
}

// Bounded wait: false when the deadline passed or another thread already aborted.
__device__ __forceinline__ bool mbar_wait_until(uint64_t* b, uint32_t parity, volatile int* abort_flag,
                                                unsigned int* err, unsigned long long timeout_ns) {
    if (mbar_try(b, parity)) return true;
    const unsigned long long t0 = global_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try(b, parity)) return true;
        if ((i & 255u) == 0u) {
            if (*abort_flag) return false;
            if (global_ns() - t0 > timeout_ns) {
                *abort_flag = 1;
                atomicOr(err, 1u);
                return false;
            }
        }
    }
}
__device__ __forceinline__ bool mbar_wait(uint64_t* b, uint32_t parity, volatile int* abort_flag,
                                          const GemmParams& p) {
    return mbar_wait_until(b, parity, abort_flag, p.err, p.timeout_ns);
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// tcgen05 shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart (stride byte offset), fixed 0b001 at bits 46-48.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)(1024u >> 4) << 32;
    d |= 1ull << 46;
    d |= 2ull << 61;  // SWIZZLE_128B
    return d;
}

// Instruction descriptor, kind::f16: fp32 accumulator, A and B both bf16 or both fp16
// (format code 1 / 0), both K-major.
__host__ __device__ constexpr uint32_t idesc_f16kind(int m, int n, bool f16) {
    return (1u << 4) | ((f16 ? 0u : 1u) << 7) | ((f16 ? 0u : 1u) << 10) | ((uint32_t)(n >> 3) << 17) |
           ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void umma_commit(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_ld16_async(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ int find_problem(const GemmParams& p, int tile) {
    int lo = 0, hi = p.nprob - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (p.prob[mid].tile_begin <= tile) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// ---------------------------------------------------------------------------------
// B = bf16 or fp16 (Hu @ q * s_t / 128) per 128-group; one warp per (token, group), for up to
// kMaxRotJobs distinct activations in one launch.  The fp32 butterfly is exact (integers
// below 2^24); the product with s_t / 128 and the bf16 conversion are the only roundings.
// ---------------------------------------------------------------------------------
struct RotJob {
    const int8_t* Xq;
    const float* scale;
    void* out;                 // bf16 or fp16 [M][K]
    int64_t first;             // first group of this job in the launch's group numbering
    int64_t groups;            // M * K / 128
    int64_t groups_per_token;  // K / 128
};
constexpr int kMaxRotJobs = 8;
struct RotParams {
    RotJob job[kMaxRotJobs];
    int njobs;
    int64_t groups;            // all jobs
};

template <bool F16>
__global__ void __launch_bounds__(256)
rotate_act_kernel16(const __grid_constant__ RotParams rp) {
    pdl_trigger();
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int64_t warp = ((int64_t)blockIdx.x * 256 + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * 256) >> 5;
    for (int64_t gg = warp; gg < rp.groups; gg += nwarps) {
        int j = 0;
        while (j + 1 < rp.njobs && rp.job[j + 1].first <= gg) ++j;
        const RotJob& jb = rp.job[j];
        const int64_t gi = gg - jb.first;
        const char4 c = *reinterpret_cast<const char4*>(jb.Xq + gi * kGroup + 4 * lane);
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
        const float sc = __ldg(jb.scale + gi / jb.groups_per_token) * (1.0f / 128.0f);
        uint2 pk;
        if constexpr (F16) {
            __half2 lo = __floats2half2_rn(v0 * sc, v1 * sc);
            __half2 hi = __floats2half2_rn(v2 * sc, v3 * sc);
            pk.x = *reinterpret_cast<uint32_t*>(&lo);
            pk.y = *reinterpret_cast<uint32_t*>(&hi);
        } else {
            __nv_bfloat162 lo = __floats2bfloat162_rn(v0 * sc, v1 * sc);
            __nv_bfloat162 hi = __floats2bfloat162_rn(v2 * sc, v3 * sc);
            pk.x = *reinterpret_cast<uint32_t*>(&lo);
            pk.y = *reinterpret_cast<uint32_t*>(&hi);
        }
        *reinterpret_cast<uint2*>(static_cast<uint16_t*>(jb.out) + gi * kGroup + 4 * lane) = pk;
    }
}

// Q4_0 activations: X [M][K] fp32 -> Xh [M][Kp] fp16, Kp = 32 ceil(K / 32), zero past K.
// Inside each group of eight k the order is 0 4 1 5 2 6 3 7, the order in which the
// dequant warps write a block's nibbles (a word's nibbles j and j + 4 share one fp16
// pair); the product sums over k, so the same order on both operands leaves it unchanged.
__global__ void __launch_bounds__(256)
q4_act_kernel(const float* __restrict__ X, int64_t K, int64_t Kp, int64_t groups,
              uint16_t* __restrict__ Xh) {
    pdl_trigger();
    pdl_wait();
    const int64_t gpt = Kp / 8;   // groups of eight per token
    for (int64_t gg = (int64_t)blockIdx.x * 256 + threadIdx.x; gg < groups;
         gg += (int64_t)gridDim.x * 256) {
        const int64_t t = gg / gpt;
        const int64_t k0 = (gg - t * gpt) * 8;
        const float* xr = X + t * K;
        float v[8];
        if (k0 + 8 <= K && (K & 3) == 0) {
            const float4 a = __ldg(reinterpret_cast<const float4*>(xr + k0));
            const float4 b = __ldg(reinterpret_cast<const float4*>(xr + k0 + 4));
            v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
            v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = (k0 + i < K) ? __ldg(xr + k0 + i) : 0.0f;
        }
        uint4 o;
        uint32_t* ow = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            __half2 h = __floats2half2_rn(v[j], v[j + 4]);
            ow[j] = *reinterpret_cast<uint32_t*>(&h);
        }
        *reinterpret_cast<uint4*>(Xh + t * Kp + k0) = o;
    }
}

// ---------------------------------------------------------------------------------
// The persistent tcgen05 GEMM.
// ---------------------------------------------------------------------------------
struct TileRef {
    int prob, mt, nt, ks;
};

__device__ __forceinline__ TileRef tile_ref(const GemmParams& p, int tile) {
    TileRef t;
    t.prob = find_problem(p, tile);
    const GemmProblem& pr = p.prob[t.prob];
    int local = tile - pr.tile_begin;
    t.ks = 0;
    if (local >= pr.tiles_per_split) {   // the second half-K tile of a split problem
        t.ks = 1;
        local -= pr.tiles_per_split;
    }
    t.mt = local % p.tiles_m;
    t.nt = local / p.tiles_m;
    return t;
}

// the stages [kb, ke) of split ks of a problem
__device__ __forceinline__ void k_range(const GemmProblem& pr, int ks, int& kb, int& ke) {
    kb = ks * pr.kchunk;
    ke = min(pr.K / kBK, kb + pr.kchunk);
}

// norm (fp16 bits) of row `o` for K-chunk `kc`, 0 for rows past N
__device__ __forceinline__ uint16_t norm_bits(const GemmProblem& pr, int o, int kc) {
    if (o >= pr.N) return 0;
    const int G = pr.K / kGroup;
    return __ldg(pr.norms + (int64_t)o * G + (kc * kBK) / kGroup);
}

__device__ __forceinline__ void umma_bf16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b,
                                                 uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate));
}

// 32-bit shared address of the pair-table entry in byte J of `wv` for this lane (table
// at a 64 KB boundary, entry e of lane l at e << 8 | l << 3): one byte permute
template <int J>
__device__ __forceinline__ uint32_t pair_addr(uint32_t wv, uint32_t lb) {
    uint32_t a;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(a) : "r"(wv), "r"(lb), "n"(0x7604 | (J << 4)));
    return a;
}
__device__ __forceinline__ uint32_t lds_u32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}
__device__ __forceinline__ float2 lds_f2(uint32_t addr) {
    float2 v;
    asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr));
    return v;
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

template <class C>
__global__ void __launch_bounds__(C::THREADS, 1) cq_gemm_kernel(const __grid_constant__ GemmParams p) {
    constexpr int kBT = C::BT;
    constexpr int kStages = C::STAGES;     // shared-memory ring = tensor-memory A ring
    constexpr int kXTileBytes = C::XTILE;
    constexpr int kStageBytes = C::STAGE;
    constexpr int kDCol0 = C::DCOL0;
    constexpr int kThreadsGemm = C::THREADS;
    constexpr int kMmaW = C::MMAW;
    constexpr int kProd = C::PROD;
    // stage barrier arrivals: one per thread that copies into the stage
    constexpr int kFullAArrivals = (kProd == 2 && C::PTILE > 0) ? 2 : 1;
    constexpr int kEpiWarp0 = C::EPI0;
    constexpr int kDequantWarp0 = C::DEQ0;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // CQ: the codeword-pair table sits at a 64 KB boundary of the shared window (the
    // address of entry e for lane l is then base | e << 8 | l << 3, one byte permute); the
    // 1024-byte aligned stages fill the space below it, then the space above it, followed
    // by the weight slabs of 1- and 3-bit rows.
    // Q4_0: no table; the stages, then the weight slabs.
    const uint32_t sbase = smem_u32(smem_raw), send = sbase + (uint32_t)kGemmSmem;
    const uint32_t a0 = (sbase + 1023u) & ~1023u;
    uint32_t tbase, b0, slab0, bars_at;
    int nA;
    if constexpr (C::FMT == kFmtCQ) {
        tbase = (sbase + 65535u) & ~65535u;
        nA = tbase >= a0 + kStageBytes ? min(kStages, (int)((tbase - a0) / kStageBytes)) : 0;
        b0 = tbase + (1u << (2 * C::BITS)) * 256u;   // the pair table: one 256-byte row per entry (32 lanes)
        slab0 = b0 + (uint32_t)(kStages - nA) * kStageBytes;
        bars_at = slab0 + (uint32_t)(C::SLABS * C::SLABBYTES);
    } else {
        tbase = 0;
        nA = kStages;
        b0 = a0;
        slab0 = a0 + (uint32_t)kStages * kStageBytes;
        bars_at = slab0 + (uint32_t)(C::SLABS * C::SLABBYTES);
    }
    auto gen = [&](uint32_t a) { return smem_raw + (a - sbase); };
    auto stage_ptr = [&](int s) {
        return gen(s < nA ? a0 + (uint32_t)s * kStageBytes : b0 + (uint32_t)(s - nA) * kStageBytes);
    };
    float2* lut2 = reinterpret_cast<float2*>(gen(tbase));   // [2^(2 BITS)][32] (CQ)
    uint64_t* bars = reinterpret_cast<uint64_t*>(gen(bars_at));
    // this CTA's tile list (problem, row tile, token tile, K half), after the barriers
    const uint32_t tiles_at = bars_at + (uint32_t)kBarBytes;
    const bool layout_ok = tiles_at + (C::TLIST ? (uint32_t)(kMaxCtaTiles * sizeof(TileRef)) : 0u) <= send;
    uint64_t* full_a = bars;                      // TMA: X tile + packed tile landed
    uint64_t* empty = bars + kStages;             // MMA: stage consumed
    uint64_t* full_b = bars + 2 * kStages;        // dequant: A stage written to TMEM
    uint64_t* acc_full = bars + 3 * kStages;      // [2] accumulator buffer ready
    uint64_t* acc_empty = acc_full + 2;           // [2] accumulator buffer drained
    uint64_t* slab_full = acc_empty + 2;          // [SLABS] weight slab landed
    uint64_t* slab_empty = slab_full + C::SLABS;  // [SLABS] slab read by the dequant of its stages
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(slab_empty + C::SLABS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    pdl_trigger();
    if (!layout_ok) {   // the launch's shared memory cannot hold the plan (host sizing error)
        if (tid == 0) atomicOr(p.err, 4u);
        return;
    }

    // codeword-pair table: entry e = (cb[e & 15], cb[e >> 4]) for 4-bit indices,
    // (cb[e & 3], cb[e >> 2]) for 2-bit ones, one copy per lane, built from the levels
    // staged in shared memory (one unrolled select per level thread)
    float* slv = reinterpret_cast<float*>(tmem_slot + 4);   // 64 bytes inside the barrier block
    if (tid < 16) {
        float v = 0.0f;
#pragma unroll
        for (int u = 0; u < 16; ++u) v = (u == tid) ? p.lv[u] : v;
        slv[tid] = v;
    }
    __syncthreads();
    if constexpr (C::HPAIR) {
        // fp16 pairs (first index low), entry e of lane l at e << 8 | l << 2
        constexpr int kHalf = C::BITS;
        constexpr int kEntries = 1 << (2 * C::BITS);
        uint32_t* luth = reinterpret_cast<uint32_t*>(gen(tbase));
        for (int i = tid; i < kEntries * 32; i += kThreadsGemm) {
            const int e = i >> 5;
            const __half2 v = __floats2half2_rn(slv[e & ((1 << kHalf) - 1)], slv[e >> kHalf]);
            luth[(e << 6) | (i & 31)] = *reinterpret_cast<const uint32_t*>(&v);
        }
    } else if constexpr (C::FMT == kFmtCQ) {
        constexpr int kHalf = C::BITS;                   // bits of one index of the pair
        constexpr int kEntries = 1 << (2 * C::BITS);
        for (int i = tid; i < kEntries * 32; i += kThreadsGemm) {
            const int e = i >> 5;
            lut2[i] = make_float2(slv[e & ((1 << kHalf) - 1)], slv[e >> kHalf]);
        }
    }
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full_a[s], kFullAArrivals);
            mbar_init(&empty[s], 1);
            mbar_init(&full_b[s], kDequantWarps);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], kMmaW);   // one commit per issuer
            mbar_init(&acc_empty[b], kEpiWarps);
        }
        for (int b = 0; b < C::SLABS; ++b) {
            mbar_init(&slab_full[b], 1);
            mbar_init(&slab_empty[b], C::SPS * kDequantWarps);   // eight warps per stage
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    // Each role walks the tiles blockIdx.x, + gridDim.x, ...; their problem lookups (a
    // binary search over the parameter block) are done here once, by all threads, so a
    // tile boundary costs one shared-memory load instead of a chain of dependent loads.
    TileRef* tlist = reinterpret_cast<TileRef*>(gen(tiles_at));
    if constexpr (C::TLIST) {
        const int ncta = (int)blockIdx.x < p.total_tiles ? (p.total_tiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
        const int nl = ncta < kMaxCtaTiles ? ncta : kMaxCtaTiles;
        for (int i = tid; i < nl; i += kThreadsGemm) tlist[i] = tile_ref(p, (int)blockIdx.x + i * (int)gridDim.x);
    }
    auto tile_at = [&](int i, int tile) {
        if constexpr (C::TLIST) return i < kMaxCtaTiles ? tlist[i] : tile_ref(p, tile);
        else return tile_ref(p, tile);
    };
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // the table, the barriers and the tensor memory are set up while the previous kernel
    // of the stream finishes; global memory is touched only after it has
    pdl_wait();

    if (warp < kProd) {
        // ------------------------------ TMA producers -----------------------------
        // one thread issues every copy, or (two producers) warp 0 the activation tiles
        // and warp 1 the packed tiles or weight slabs; a thread with no copy in a stage
        // still walks it, to keep its ring position
        if (lane == 0) {
            const bool cx = warp == 0;                    // activation tiles
            const bool cp = warp == kProd - 1;            // packed tiles and slabs
            int s = 0;
            uint32_t ph = 0;
            bool ok = true;
            int pg = 0;   // slabs issued
            int ti = 0;
            for (int tile = blockIdx.x; ok && tile < p.total_tiles; tile += gridDim.x, ++ti) {
                const TileRef tr = tile_at(ti, tile);
                const GemmProblem& pr = p.prob[tr.prob];
                const CUtensorMap* xmap = &p.tmap[pr.act];
                int kb, ke;
                k_range(pr, tr.ks, kb, ke);
                for (int kc = kb; kc < ke; ++kc) {
                    if constexpr (C::SLABS > 0) {
                        // the slab of this stage and the next SPS - 1 (tile K ranges are
                        // whole slabs)
                        if (cp && kc % C::SPS == 0) {
                            const int qs = pg % C::SLABS;
                            const uint32_t sph = (uint32_t)((pg / C::SLABS) & 1);
                            if (!mbar_wait(&slab_empty[qs], sph ^ 1u, abort_flag, p)) {
                                ok = false;
                                break;
                            }
                            mbar_arrive_tx(&slab_full[qs], C::SLABBYTES);
                            tma_load_2d(gen(slab0 + (uint32_t)(qs * C::SLABBYTES)), &pr.pmap,
                                        (kc / C::SPS) * C::SLABROW, tr.nt * kBO, &slab_full[qs]);
                            ++pg;
                        }
                    }
                    if (cx || (cp && C::PTILE > 0)) {
                        if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag, p)) { ok = false; break; }
                        uint8_t* st = stage_ptr(s);
                        if (cx) {
                            // with one producer the packed tile rides on the same arrival
                            const uint32_t bytes = kXTileBytes + (kProd == 1 ? (uint32_t)C::PTILE : 0u);
                            mbar_arrive_tx(&full_a[s], bytes);
                            tma_load_2d(st, xmap, kc * kBK, tr.mt * kBT, &full_a[s]);
                        } else {
                            mbar_arrive_tx(&full_a[s], (uint32_t)C::PTILE);
                        }
                        if constexpr (C::PTILE > 0) {
                            if (cp)
                                tma_load_2d(st + kXTileBytes, &pr.pmap, kc * (kBK * C::BITS / 8), tr.nt * kBO,
                                            &full_a[s]);
                        }
                    }
                    if (++s == kStages) { s = 0; ph ^= 1u; }
                }
            }
        }
        __syncwarp();
    } else if (warp < kProd + kMmaW) {
        // ------------------------------ MMA issuers -------------------------------
        // issuer mj takes the stages t of each tile with t % kMmaW == mj (all of them when
        // there is one issuer) into its partial accumulator of the tile's buffer
        if (lane == 0) {
            const int mj = warp - kProd;
            constexpr uint32_t idesc = idesc_f16kind(kBO, kBT, C::OPF16);
            int s = 0, sa = 0;   // shared stage, A stage
            uint32_t pha = 0;
            int it = 0;
            bool ok = true;
            // B descriptors differ only in the low word (the 16-byte-unit stage address):
            // kept as a running value, stepped per stage, jumping over the pair table
            const uint64_t dhi = smem_desc_sw128(0u);
            const uint32_t lo_first = (uint32_t)smem_desc_sw128(smem_u32(stage_ptr(0)));
            const uint32_t lo_above = (uint32_t)smem_desc_sw128(smem_u32(stage_ptr(nA < kStages ? nA : 0)));
            uint32_t blo = lo_first;
            uint32_t aaddr = tmem_base;   // A stage sa
            for (int tile = blockIdx.x; ok && tile < p.total_tiles; tile += gridDim.x, ++it) {
                const TileRef tr = tile_at(it, tile);
                const GemmProblem& pr = p.prob[tr.prob];
                const int buf = it & 1;
                const uint32_t aph = (uint32_t)((it >> 1) & 1);
                int kb, ke;
                k_range(pr, tr.ks, kb, ke);
                // every issuer waits for the buffer, also one without a stage in this tile
                // (its partial stays unwritten; the epilogue adds only the partials of the
                // tile's first kMmaW stages): its acc_full commit then cannot arrive on the
                // barrier before the buffer's previous phase has completed
                if (!mbar_wait(&acc_empty[buf], aph ^ 1u, abort_flag, p)) break;
                tc_fence_after();
                const uint32_t d = tmem_base + (uint32_t)(kDCol0 + (buf * kMmaW + mj) * kBT);
                for (int kc = kb; kc < ke; ++kc) {
                    if ((kc - kb) % kMmaW == mj) {
                        // the dequant warps arrive on full_b only after waiting on the TMA
                        // barrier of the same stage, so it also orders the TMA writes
                        if (!mbar_wait(&full_b[sa], pha, abort_flag, p)) { ok = false; break; }
                        tc_fence_after();
#pragma unroll
                        for (int kk = 0; kk < kBK / 16; ++kk) {
                            // A: 8 TMEM columns (16 bf16) per K step; B: +32 bytes along K
                            // inside the swizzle atom = +2 in the 16-byte-unit address field
                            umma_bf16_tmem_a(d, aaddr + (uint32_t)(8 * kk), dhi | (uint64_t)(blo + 2u * kk), idesc,
                                             (kc - kb >= kMmaW || kk > 0) ? 1u : 0u);
                        }
                        umma_commit(&empty[s]);
                    }
                    ++s;
                    blo += (uint32_t)(kStageBytes >> 4);
                    if (s == nA) blo = lo_above;
                    if (s == kStages) { s = 0; blo = lo_first; }
                    aaddr += (uint32_t)kACols;
                    if (++sa == kStages) { sa = 0; pha ^= 1u; aaddr = tmem_base; }
                }
                if (!ok) break;
                umma_commit(&acc_full[buf]);
            }
        }
        __syncwarp();
    } else if (warp < kDequantWarp0) {
        // ------------------------------ epilogue ----------------------------------
        // warp -> TMEM lane quarter q (out-rows 32q..32q+31) and token slice th of kTW
        // tokens (96 of the prefill's 192 with eight epilogue warps)
        constexpr int kTW = kBT / (kEpiWarps / 4);
        const int q = warp & 3;
        const int th = (warp - kEpiWarp0) >> 2;
        int it = 0;
        for (int tile = blockIdx.x; tile < p.total_tiles; tile += gridDim.x, ++it) {
            const TileRef tr = tile_at(it, tile);
            const GemmProblem& pr = p.prob[tr.prob];
            const int buf = it & 1;
            if (!mbar_wait(&acc_full[buf], (uint32_t)((it >> 1) & 1), abort_flag, p)) break;
            tc_fence_after();
            const uint32_t col0 = tmem_base + ((uint32_t)(q * 32) << 16) +
                                  (uint32_t)(kDCol0 + buf * kMmaW * kBT + th * kTW);
            const int o = tr.nt * kBO + q * 32 + lane;
            const int t0 = tr.mt * kBT + th * kTW;
            const bool ook = o < pr.N;
            __nv_bfloat16* ycol = static_cast<__nv_bfloat16*>(pr.Y) + o;
            float* ycolf = static_cast<float*>(pr.Y) + o;
            // 16-column pieces, each load issued before the previous piece is stored
            constexpr int kPieces = kTW / 16;
            uint32_t rr[2][16];
            auto store16 = [&](const uint32_t (&r)[16], int tb) {
                if (!ook) return;
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int t = tb + j;
                    if (t < p.M) {
                        if constexpr (C::F16) {
                            if (pr.ksplit > 1) atomicAdd(ycolf + (int64_t)t * pr.N, __uint_as_float(r[j]));
                            else ycolf[(int64_t)t * pr.N] = __uint_as_float(r[j]);
                        } else {
                            ycol[(int64_t)t * pr.N] = __float2bfloat16_rn(__uint_as_float(r[j]));
                        }
                    }
                }
            };
            if constexpr (kMmaW == 1) {
                tmem_ld16_async(col0, rr[0]);
#pragma unroll
                for (int pc = 0; pc < kPieces; ++pc) {
                    tmem_wait_ld();
                    if (pc + 1 < kPieces) tmem_ld16_async(col0 + 16 * (pc + 1), rr[(pc + 1) & 1]);
                    store16(rr[pc & 1], t0 + 16 * pc);
                }
            } else {
                // per 16-column piece, the partials of the issuers that had a stage in this
                // tile, summed in issuer order
                int kb, ke;
                k_range(pr, tr.ks, kb, ke);
                const int np = min(kMmaW, ke - kb);
#pragma unroll
                for (int pc = 0; pc < kPieces; ++pc) {
                    tmem_ld16_async(col0 + 16 * pc, rr[0]);
                    tmem_wait_ld();
                    for (int j = 1; j < np; ++j) {
                        tmem_ld16_async(col0 + (uint32_t)(j * kBT + 16 * pc), rr[1]);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            rr[0][i] = __float_as_uint(__uint_as_float(rr[0][i]) + __uint_as_float(rr[1][i]));
                    }
                    store16(rr[0], t0 + 16 * pc);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[buf]);
        }
    } else {
        // ------------------------------ dequant -----------------------------------
        // warp -> TMEM lane quarter q (out-rows 32q..32q+31), k half kh (32 of the 64 k of
        // a stage) and stage group grp; lane -> one row: 16 packed bytes -> 16 codeword
        // pairs (one table lookup each) x norm -> bf16 pairs -> tcgen05.st of 16 columns
        const int dw = warp - kDequantWarp0;
        const int q = warp & 3;
        const int kh = (dw >> 2) & 1;
        const int grp = dw >> 3;
        const int r = q * 32 + lane;
        const uint32_t lb = tbase | ((uint32_t)lane << 3);
        bool ok = true;
        int gi = 0;   // global stage index
        int ti = 0;
        // this lane's row norms, eight (16 bytes) or four groups (8 bytes) per load where
        // the rows allow it: one scattered 2-byte load per lane and stage made the norms
        // the largest consumer of the L1 data pipe
        uint4 nv = make_uint4(0u, 0u, 0u, 0u);
        int nv_g0 = -1;   // first group held in nv, -1: none
        for (int tile = blockIdx.x; ok && tile < p.total_tiles; tile += gridDim.x, ++ti) {
            const TileRef tr = tile_at(ti, tile);
            const GemmProblem& pr = p.prob[tr.prob];
            int kb, ke;
            k_range(pr, tr.ks, kb, ke);
            const int orow = tr.nt * kBO + r;
            const int G = pr.K / kGroup;
            const uintptr_t nal = reinterpret_cast<uintptr_t>(pr.norms);
            const int nvw = ((G & 7) == 0 && (nal & 15u) == 0) ? 8 : ((G & 3) == 0 && (nal & 7u) == 0) ? 4 : 0;
            nv_g0 = -1;
            for (int kc = kb; kc < ke; ++kc, ++gi) {
                if (gi % kDequantGroups != grp) continue;   // the other group's stage
                const int s = gi % kStages;
                const uint32_t ph = (uint32_t)((gi / kStages) & 1);
                const int sa = s;   // the A stage in tensor memory (the copy of the same stage
                                    // landing implies its previous MMA has completed)
                if constexpr (C::FMT == kFmtQ40) {
                    // the full_a wait frees the A stage (its previous MMA has completed)
                    // and, through full_b, orders the activation tile for the MMA
                    if (!mbar_wait(&full_a[s], ph, abort_flag, p)) { ok = false; break; }
                    const int sg = gi / C::SPS;   // every K is a whole number of slabs
                    const int qs = sg % C::SLABS;
                    if (!mbar_wait(&slab_full[qs], (uint32_t)((sg / C::SLABS) & 1), abort_flag, p)) {
                        ok = false;
                        break;
                    }
                    // block (kc & 3) * 2 + kh of this row's 144-byte slab row starts at
                    // byte 36 (kc & 3) + 18 kh: five words from the 4-byte boundary at or
                    // below it hold the fp16 scale and the 16 nibble bytes
                    const uint32_t* w32 = reinterpret_cast<const uint32_t*>(
                        gen(slab0 + (uint32_t)(qs * C::SLABBYTES) + (uint32_t)(r * C::SLABROW)));
                    const int wb = 9 * (kc & 3) + 4 * kh;
                    uint32_t w[5];
#pragma unroll
                    for (int i = 0; i < 5; ++i) w[i] = w32[wb + i];
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&slab_empty[qs]);
                    uint32_t d2;   // the scale in both halves
                    asm("prmt.b32 %0, %1, 0, %2;" : "=r"(d2) : "r"(w[0]), "r"(kh ? 0x3232u : 0x1010u));
                    const __half2 hd = *reinterpret_cast<const __half2*>(&d2);
                    const __half2 bias = __halves2half2(__ushort_as_half((unsigned short)0x6408u),
                                                        __ushort_as_half((unsigned short)0x6408u));
                    const uint32_t sh = kh ? 32u : 16u;
                    uint32_t pk[16];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        // nibbles 0..7 of this word are the block's elements 8i..8i+7;
                        // output word 4i + j holds elements (8i + j, 8i + j + 4), each as
                        // 1024 + nib in fp16, minus 1032, times d
                        const uint32_t qw = __funnelshift_rc(w[i], w[i + 1], sh);
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const uint32_t v = ((qw >> (4 * j)) & 0x000F000Fu) | 0x64006400u;
                            __half2 h = __hsub2(*reinterpret_cast<const __half2*>(&v), bias);
                            h = __hmul2(h, hd);
                            pk[4 * i + j] = *reinterpret_cast<uint32_t*>(&h);
                        }
                    }
                    tmem_st16(tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(sa * kACols + kh * 16), pk);
                    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&full_b[sa]);
                    continue;
                }
                uint16_t nb;
                if (nvw != 0) {
                    const int g = (kc * kBK) / kGroup;
                    if ((g & -nvw) != nv_g0) {
                        nv_g0 = g & -nvw;
                        const uint16_t* src = pr.norms + (int64_t)orow * G + nv_g0;
                        if (orow >= pr.N) {
                            nv = make_uint4(0u, 0u, 0u, 0u);
                        } else if (nvw == 8) {
                            nv = __ldg(reinterpret_cast<const uint4*>(src));
                        } else {
                            const uint2 h = __ldg(reinterpret_cast<const uint2*>(src));
                            nv = make_uint4(h.x, h.y, 0u, 0u);
                        }
                    }
                    const int j = g & (nvw - 1);
                    const uint32_t w = (j >> 1) == 0 ? nv.x : (j >> 1) == 1 ? nv.y : (j >> 1) == 2 ? nv.z : nv.w;
                    nb = (uint16_t)(w >> ((j & 1) * 16));
                } else {
                    nb = norm_bits(pr, orow, kc);
                }
                if (!mbar_wait(&full_a[s], ph, abort_flag, p)) { ok = false; break; }
                if constexpr (C::CQSLAB) {
                    const int sg = gi / C::SPS;   // every K is a whole number of slabs
                    const int qs = sg % C::SLABS;
                    if (!mbar_wait(&slab_full[qs], (uint32_t)((sg / C::SLABS) & 1), abort_flag, p)) {
                        ok = false;
                        break;
                    }
                    // half kh of stage kc & 1 starts at index 64 (kc & 1) + 32 kh of the
                    // slab row: BITS whole words (the rows are LSB-first bit strings)
                    const uint32_t* w32 = reinterpret_cast<const uint32_t*>(
                        gen(slab0 + (uint32_t)(qs * C::SLABBYTES) + (uint32_t)(r * C::SLABROW)));
                    const int wb = ((kc & 1) * 2 + kh) * C::BITS;
                    uint32_t w[C::BITS + 1];
#pragma unroll
                    for (int i = 0; i < C::BITS; ++i) w[i] = w32[wb + i];
                    w[C::BITS] = 0u;
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&slab_empty[qs]);
                    const float nrm = f16_bits_to_f32(nb);
                    const float2 n2 = make_float2(nrm, nrm);
                    uint32_t pk[16];
#pragma unroll
                    for (int pi = 0; pi < 16; ++pi) {
                        // pair pi = indices 2 pi, 2 pi + 1: 2 BITS bits from bit 2 BITS pi
                        constexpr int kPB = 2 * C::BITS;
                        const int bo = kPB * pi;
                        const uint32_t v = __funnelshift_r(w[bo >> 5], w[(bo >> 5) + 1], bo & 31);
                        const uint32_t e = v & ((1u << kPB) - 1u);
                        const float2 cn = __fmul2_rn(lds_f2(lb + (e << 8)), n2);
                        __half2 h = __floats2half2_rn(cn.x, cn.y);
                        pk[pi] = *reinterpret_cast<uint32_t*>(&h);
                    }
                    tmem_st16(tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(sa * kACols + kh * 16), pk);
                    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&full_b[sa]);
                    continue;
                }
                // this lane's 32 indices of the stage half kh, as 16 pair bytes: 4-bit rows
                // hold one pair per byte; a 2-bit byte holds two pairs, split by nibble
                // (the low nibble is the byte's first pair)
                uint32_t wv[4];
                if constexpr (C::BITS == 4) {
                    const uint4 w = *reinterpret_cast<const uint4*>(stage_ptr(s) + kXTileBytes + r * 32 + kh * 16);
                    wv[0] = w.x; wv[1] = w.y; wv[2] = w.z; wv[3] = w.w;
                } else {
                    const uint2 w = *reinterpret_cast<const uint2*>(stage_ptr(s) + kXTileBytes + r * 16 + kh * 8);
                    wv[0] = w.x & 0x0F0F0F0Fu; wv[1] = (w.x >> 4) & 0x0F0F0F0Fu;
                    wv[2] = w.y & 0x0F0F0F0Fu; wv[3] = (w.y >> 4) & 0x0F0F0F0Fu;
                }
                uint32_t pk[16];
                if constexpr (C::HPAIR) {
                    // fp16 pair lookups (4 bytes) times the fp16 norm (exact: the norm is
                    // stored as fp16): one multiply per pair, no conversion
                    const uint32_t lb4 = tbase | ((uint32_t)lane << 2);
                    const __half2 nh = __halves2half2(__ushort_as_half(nb), __ushort_as_half(nb));
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const uint32_t c[4] = {lds_u32(pair_addr<0>(wv[k], lb4)), lds_u32(pair_addr<1>(wv[k], lb4)),
                                               lds_u32(pair_addr<2>(wv[k], lb4)), lds_u32(pair_addr<3>(wv[k], lb4))};
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            // pair index within the half: byte j of word k (4-bit), or byte j
                            // of packed word k / 2, low or high nibble (2-bit)
                            const int pi = C::BITS == 4 ? 4 * k + j : 8 * (k >> 1) + 2 * j + (k & 1);
                            const __half2 v = __hmul2(*reinterpret_cast<const __half2*>(&c[j]), nh);
                            pk[pi] = *reinterpret_cast<const uint32_t*>(&v);
                        }
                    }
                    tmem_st16(tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(sa * kACols + kh * 16), pk);
                    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&full_b[sa]);
                    continue;
                }
                const float nrm = f16_bits_to_f32(nb);
                const float2 n2 = make_float2(nrm, nrm);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float2 c[4] = {lds_f2(pair_addr<0>(wv[k], lb)), lds_f2(pair_addr<1>(wv[k], lb)),
                                         lds_f2(pair_addr<2>(wv[k], lb)), lds_f2(pair_addr<3>(wv[k], lb))};
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        // pair index within the half: byte j of word k (4-bit), or byte j
                        // of packed word k / 2, low or high nibble (2-bit)
                        const int pi = C::BITS == 4 ? 4 * k + j : 8 * (k >> 1) + 2 * j + (k & 1);
                        const float2 cn = __fmul2_rn(c[j], n2);
                        if constexpr (C::F16) {
                            __half2 v = __floats2half2_rn(cn.x, cn.y);
                            pk[pi] = *reinterpret_cast<uint32_t*>(&v);
                        } else {
                            __nv_bfloat162 v = __floats2bfloat162_rn(cn.x, cn.y);
                            pk[pi] = *reinterpret_cast<uint32_t*>(&v);
                        }
                    }
                }
                tmem_st16(tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(sa * kACols + kh * 16), pk);
                asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&full_b[sa]);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                     "r"(kTmemCols));
    }
}

// ---------------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------------
static __device__ unsigned int g_gemm_err;

std::mutex g_host_mu;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
unsigned int* g_err_ptr[64] = {nullptr};
bool g_attr_done[64][7] = {};

template <class C>
cq_status set_smem_attr(int dev, int slot) {
    if (g_attr_done[dev][slot]) return CQ_OK;
    const cudaError_t e = cudaFuncSetAttribute(cq_gemm_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               kGemmSmem);
    if (e != cudaSuccess) { set_last_cuda_error((int)e); return CQ_ERR_CUDA; }
    g_attr_done[dev][slot] = true;
    return CQ_OK;
}

cq_status host_setup(unsigned int** err) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) { set_last_cuda_error((int)e); return CQ_ERR_CUDA; }
    if (dev < 0 || dev >= 64) return CQ_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_host_mu);
    if (!g_encode) {
        cudaDriverEntryPointQueryResult q;
        void* fn = nullptr;
        e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) {
            set_last_cuda_error((int)e);
            return CQ_ERR_UNSUPPORTED;
        }
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    if (!g_err_ptr[dev]) {
        void* pe = nullptr;
        e = cudaGetSymbolAddress(&pe, g_gemm_err);
        if (e != cudaSuccess) { set_last_cuda_error((int)e); return CQ_ERR_CUDA; }
        g_err_ptr[dev] = static_cast<unsigned int*>(pe);
    }
    cq_status st = set_smem_attr<PrefillCfg>(dev, 0);
    if (st == CQ_OK) st = set_smem_attr<DecodeCfg>(dev, 1);
    if (st == CQ_OK) st = set_smem_attr<Q40WideCfg>(dev, 2);
    if (st == CQ_OK) st = set_smem_attr<Q40NarrowCfg>(dev, 3);
    if (st == CQ_OK) st = set_smem_attr<Decode2Cfg>(dev, 4);
    if (st == CQ_OK) st = set_smem_attr<Decode1Cfg>(dev, 5);
    if (st == CQ_OK) st = set_smem_attr<Decode3Cfg>(dev, 6);
    if (st != CQ_OK) return st;
    *err = g_err_ptr[dev];
    return CQ_OK;
}

// Encoded weight maps by (address, N, K): a map depends on nothing else, so a cached one
// stays valid for any tensor later placed at the same address with the same shape.
// Guarded by g_host_mu (held by the caller).
struct MapEntry {
    const void* base;
    int64_t N, K;
    int bits;
    CUtensorMap map;
};
constexpr int kMapCache = 4096;   // power of two
MapEntry g_map_cache[kMapCache];

cq_status make_packed_map_uncached(CUtensorMap* map, const void* base, int64_t N, int64_t K, int bits);

cq_status make_packed_map(CUtensorMap* map, const void* base, int64_t N, int64_t K, int bits) {
    uint64_t h = reinterpret_cast<uint64_t>(base) * 0x9E3779B97F4A7C15ull ^ (uint64_t)N * 0xC2B2AE3D27D4EB4Full ^
                 ((uint64_t)K << 3 | (uint64_t)bits);
    for (int probe = 0; probe < 8; ++probe) {
        MapEntry& e = g_map_cache[(h + (uint64_t)probe) & (kMapCache - 1)];
        if (e.base == base && e.N == N && e.K == K && e.bits == bits) {
            *map = e.map;
            return CQ_OK;
        }
        if (e.base == nullptr) {
            const cq_status st = make_packed_map_uncached(&e.map, base, N, K, bits);
            if (st != CQ_OK) return st;
            e.base = base; e.N = N; e.K = K; e.bits = bits;
            *map = e.map;
            return CQ_OK;
        }
    }
    return make_packed_map_uncached(map, base, N, K, bits);   // neighbourhood full: no caching
}

// packed index rows [N][K * bits / 8] bytes; box = one stage's kBK indices x 128 rows
// (32 bytes for 4-bit rows, 16 for 2-bit ones), or a slab of two stages for 1- and 3-bit
// rows (16 and 48 bytes)
cq_status make_packed_map_uncached(CUtensorMap* map, const void* base, int64_t N, int64_t K, int bits) {
    const int box_k = (bits == 1 || bits == 3) ? 2 * kBK : kBK;
    cuuint64_t dims[2] = {(cuuint64_t)(K * bits / 8), (cuuint64_t)N};
    cuuint64_t strides[1] = {(cuuint64_t)(K * bits / 8)};
    cuuint32_t box[2] = {(cuuint32_t)(box_k * bits / 8), (cuuint32_t)kBO};
    cuuint32_t estr[2] = {1u, 1u};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) { set_last_cuda_error((int)r); return CQ_ERR_CUDA; }
    return CQ_OK;
}

// Q4_0 block rows [N][nblk * 18] bytes (nblk a multiple of 8), box = one 144-byte slab
// row (8 blocks) x 128 rows
cq_status make_q40_map(CUtensorMap* map, const void* base, int64_t N, int64_t nblk) {
    const cuuint64_t rowbytes = (cuuint64_t)nblk * 18u;
    cuuint64_t dims[2] = {rowbytes, (cuuint64_t)N};
    cuuint64_t strides[1] = {rowbytes};
    cuuint32_t box[2] = {(cuuint32_t)kQSlabRowBytes, (cuuint32_t)kBO};
    cuuint32_t estr[2] = {1u, 1u};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) { set_last_cuda_error((int)r); return CQ_ERR_CUDA; }
    return CQ_OK;
}

cq_status make_act_map(CUtensorMap* map, const void* base, int64_t M, int64_t K, int bt, bool f16) {
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
    cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)bt};
    cuuint32_t estr[2] = {1u, 1u};
    CUresult r = g_encode(map, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                          const_cast<void*>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) { set_last_cuda_error((int)r); return CQ_ERR_CUDA; }
    return CQ_OK;
}

// K split of one problem.  The 32-token configurations reach one weight tile per ~120
// cycles of MMA issue per SM, so every SM should hold tiles: when the output tiles alone
// number under 1.5 per SM, each is cut into two half-K tiles (a multiple of `align`
// stages) whose fp32 partials the epilogue adds into Y.  Two addends on a zeroed Y give
// the same sum in either order, so results stay bit-reproducible.
template <class C>
void choose_split(GemmProblem& gp, int tiles_m, int align) {
    const int nk = gp.K / kBK;
    gp.tiles_per_split = gp.tiles_n * tiles_m;
    gp.ksplit = 1;
    gp.kchunk = nk;
    if (C::F16 && C::BT == 32 && 2 * gp.tiles_per_split <= 3 * sm_count() && nk >= 2 * align) {
        int chunk = (nk + 1) / 2;
        chunk = (chunk + align - 1) / align * align;
        if (chunk < nk) {
            gp.ksplit = 2;
            gp.kchunk = chunk;
        }
    }
}

}  // namespace

// Failure-detection probe for the pipeline's wait: one thread waits on a barrier phase that
// nothing completes; after p.timeout_ns the wait raises the abort flag and the error word
// and returns (the path every role of cq_gemm_kernel takes when a wait runs out).
__global__ void bounded_wait_probe_gemm_kernel(unsigned int* err, unsigned long long timeout_ns) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (threadIdx.x == 0) (void)mbar_wait_until(&bar, 0u, &abort_flag, err, timeout_ns);
}

cq_status probe_gemm_wait(unsigned long long timeout_ns, cudaStream_t st) {
    unsigned int* err = nullptr;
    const cq_status se = host_setup(&err);
    if (se != CQ_OK) return se;
    bounded_wait_probe_gemm_kernel<<<1, 32, 0, st>>>(err, timeout_ns);
    return check_launch();
}

unsigned int* gemm_error_word(int dev) {
    if (dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(g_host_mu);
    return g_err_ptr[dev];
}

}  // namespace cq

using namespace cq;

extern "C" size_t cq_gemm_workspace_bytes(int64_t M, int64_t K) {
    if (M < 1 || K < 1) return 0;
    return ((size_t)M * (size_t)K * 2u + 255u) & ~(size_t)255u;
}

extern "C" size_t cq_gemm_grouped_workspace_bytes(const cq_gemm_problem* probs, int count, int64_t M) {
    if (!probs || count < 1 || M < 1) return 0;
    size_t total = 0;
    for (int i = 0; i < count; ++i) {
        bool seen = false;
        for (int j = 0; j < i; ++j)
            if (probs[j].Xq == probs[i].Xq) { seen = true; break; }
        if (!seen) total += ((size_t)M * (size_t)probs[i].K * 2u + 255u) & ~(size_t)255u;
    }
    return total;
}

// The launch sequence shared by the prefill GEMM and the batched decode product: the
// distinct activations are rotated into the workspace, then the problems go out in
// launches of at most kMaxProblems problems and kMaxActs activations each.  The caller
// has validated the problems and the workspace.  Each problem's Y is bf16 (prefill) or
// fp32 (decode, C::F16).
template <class C>
cq_status run_grouped(const cq_gemm_problem* probs, int count, int64_t M, int b,
                      const cq_codebook* cbk, void* workspace, cudaStream_t cs) {
    // tile numbers are 32-bit: a problem may hold up to 2^23 output tiles (twice that
    // when split), so a launch of kMaxProblems problems stays below 2^31
    const int64_t tiles_m64 = (M + C::BT - 1) / C::BT;
    for (int i = 0; i < count; ++i)
        if (tiles_m64 * ((probs[i].N + kBO - 1) / kBO) > ((int64_t)1 << 23)) return CQ_ERR_UNSUPPORTED;
    unsigned int* err = nullptr;
    cq_status st = host_setup(&err);
    if (st != CQ_OK) return st;

    // distinct activations -> rotated 16-bit copies in the workspace, up to kMaxRotJobs
    // activations per rotation launch
    if (count > 1024) return CQ_ERR_UNSUPPORTED;
    const int8_t* act_src[1024];
    const void* act_dst[1024];
    int64_t act_K[1024];
    int act_of[1024];
    int nact = 0;
    size_t off = 0;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    RotParams rp;
    rp.njobs = 0;
    rp.groups = 0;
    auto flush_rot = [&]() -> cq_status {
        if (rp.njobs == 0) return CQ_OK;
        int64_t grid = (rp.groups + 7) / 8;
        const int64_t cap = (int64_t)sm_count() * 16;
        if (grid > cap) grid = cap;
        const cq_status r = launch_pdl(rotate_act_kernel16<C::OPF16>, dim3((unsigned)grid), dim3(256), 0, cs, rp);
        rp.njobs = 0;
        rp.groups = 0;
        return r;
    };
    for (int i = 0; i < count; ++i) {
        int a = -1;
        for (int j = 0; j < nact; ++j)
            if (act_src[j] == probs[i].Xq) { a = j; break; }
        if (a < 0) {
            a = nact++;
            act_src[a] = probs[i].Xq;
            act_dst[a] = ws + off;
            act_K[a] = probs[i].K;
            if (rp.njobs == kMaxRotJobs) {
                st = flush_rot();
                if (st != CQ_OK) return st;
            }
            RotJob& jb = rp.job[rp.njobs++];
            jb.Xq = probs[i].Xq;
            jb.scale = probs[i].scale;
            jb.out = ws + off;
            jb.first = rp.groups;
            jb.groups_per_token = probs[i].K / kGroup;
            jb.groups = M * jb.groups_per_token;
            rp.groups += jb.groups;
            off += ((size_t)M * (size_t)probs[i].K * 2u + 255u) & ~(size_t)255u;
        }
        act_of[i] = a;
    }
    st = flush_rot();
    if (st != CQ_OK) return st;

    // launches of at most kMaxProblems problems and kMaxActs activations each, larger K
    // first so the long tiles start early
    int order[1024];
    for (int i = 0; i < count; ++i) order[i] = i;
    for (int i = 1; i < count; ++i) {
        const int v = order[i];
        int j = i - 1;
        while (j >= 0 && probs[order[j]].K < probs[v].K) { order[j + 1] = order[j]; --j; }
        order[j + 1] = v;
    }
    static GemmParams prm;   // large; built on the host, passed by value to the launch
    std::lock_guard<std::mutex> lock(g_host_mu);
    int i0 = 0;
    while (i0 < count) {
        memset(&prm, 0, sizeof(prm));
        int map_of_act[1024];
        for (int a = 0; a < nact; ++a) map_of_act[a] = -1;
        int nmaps = 0, np = 0, tiles = 0;
        const int tiles_m = (int)((M + C::BT - 1) / C::BT);
        while (i0 < count && np < kMaxProblems) {
            const int pi = order[i0];
            const int a = act_of[pi];
            if (map_of_act[a] < 0) {
                if (nmaps == kMaxActs) break;
                st = make_act_map(&prm.tmap[nmaps], act_dst[a], M, act_K[a], C::BT, C::OPF16);
                if (st != CQ_OK) return st;
                map_of_act[a] = nmaps++;
            }
            const cq_gemm_problem& q = probs[pi];
            GemmProblem& gp = prm.prob[np++];
            gp.packed = q.packed; gp.norms = q.norms; gp.scale = q.scale;
            gp.Y = q.Y;
            gp.N = (int)q.N; gp.K = (int)q.K; gp.act = map_of_act[a];
            st = make_packed_map(&gp.pmap, q.packed, q.N, q.K, C::BITS);
            if (st != CQ_OK) return st;
            gp.tiles_n = (int)((q.N + kBO - 1) / kBO);
            gp.tile_begin = tiles;
            choose_split<C>(gp, tiles_m, C::SLABS > 0 ? C::SPS : 1);   // whole slabs
            if (gp.ksplit > 1) {
                const cudaError_t e = cudaMemsetAsync(q.Y, 0, (size_t)M * (size_t)q.N * sizeof(float), cs);
                if (e != cudaSuccess) { set_last_cuda_error((int)e); return CQ_ERR_CUDA; }
            }
            tiles += gp.tiles_per_split * gp.ksplit;
            ++i0;
        }
        prm.nprob = np;
        prm.M = (int)M;
        prm.tiles_m = tiles_m;
        prm.total_tiles = tiles;
        cq_host_levels(prm.lv, b, cbk);
        prm.err = err;
        prm.timeout_ns = 2000000000ull;   // 2 s per wait
        const size_t smem = (size_t)kGemmSmem;
        const int grid = tiles < sm_count() ? tiles : sm_count();
        st = launch_pdl(cq_gemm_kernel<C>, dim3(grid), dim3(C::THREADS), smem, cs, prm);
        if (st != CQ_OK) return st;
    }
    return CQ_OK;
}


extern "C" cq_status cq_gemm_grouped(const cq_gemm_problem* probs, int count, int64_t M, int g,
                                     int b, const cq_codebook* cbk, void* workspace,
                                     size_t workspace_bytes, void* stream) {
    if (!probs || count < 1 || !cbk || M < 1 || M > (1 << 30)) return CQ_ERR_INVALID_ARG;
    if (g != kGroup || !cq_code_valid(b)) return CQ_ERR_INVALID_ARG;
    if (b != 4) return CQ_ERR_UNSUPPORTED;
    for (int i = 0; i < count; ++i) {
        const cq_gemm_problem& q = probs[i];
        if (!q.packed || !q.norms || !q.Xq || !q.scale || !q.Y) return CQ_ERR_INVALID_ARG;
        if (q.N < 1 || q.K < kGroup || q.K % kGroup != 0 || q.N % 16 != 0 || q.K > (1 << 24) ||
            q.N > (1 << 24))
            return CQ_ERR_INVALID_ARG;
        if (!aligned16(q.packed) || !aligned16(q.norms) || !aligned16(q.Xq) ||
            !aligned16(q.scale) || !aligned16(q.Y))
            return CQ_ERR_ALIGNMENT;
        for (int j = 0; j < i; ++j)
            if (probs[j].Xq == q.Xq && probs[j].K != q.K) return CQ_ERR_INVALID_ARG;
    }
    const size_t need = cq_gemm_grouped_workspace_bytes(probs, count, M);
    if (!workspace || workspace_bytes < need) return CQ_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return CQ_ERR_ALIGNMENT;

    return run_grouped<PrefillCfg>(probs, count, M, b, cbk, workspace, as_stream(stream));
}

extern "C" cq_status cq_gemm(const uint8_t* packed, const uint16_t* norms, int64_t N, int64_t K,
                             int g, int b, const cq_codebook* cbk, const int8_t* Xq,
                             const float* scale, int64_t M, uint16_t* Y, void* workspace,
                             size_t workspace_bytes, void* stream) {
    cq_gemm_problem q;
    q.packed = packed; q.norms = norms; q.N = N; q.K = K; q.Xq = Xq; q.scale = scale; q.Y = Y;
    if (workspace_bytes < cq_gemm_workspace_bytes(M, K)) return CQ_ERR_WORKSPACE;
    return cq_gemm_grouped(&q, 1, M, g, b, cbk, workspace, workspace_bytes, stream);
}


namespace cq {

// The batched decode product of cq_gemv (1- to 4-bit indices) on the tensor cores: the
// same pipeline with 32-token tiles, fp16 operands (so the result meets the fp32 GEMV's
// error bound) and fp32 output.  `workspace` (16-byte aligned, at least B * K * 2 + 256
// bytes) receives the rotated fp16 activations.
cq_status gemv_tensor(const uint8_t* packed, const uint16_t* norms, int64_t N, int64_t K, int b,
                      const cq_codebook* cbk, const int8_t* Xq, const float* scale, int64_t B,
                      float* Y, void* workspace, cudaStream_t st) {
    cq_gemm_problem q;
    q.packed = packed; q.norms = norms; q.N = N; q.K = K; q.Xq = Xq; q.scale = scale;
    q.Y = reinterpret_cast<uint16_t*>(Y);   // the pipeline stores fp32 for this configuration
    switch (b) {
        case 1: return run_grouped<Decode1Cfg>(&q, 1, B, 1, cbk, workspace, st);
        case 2: return run_grouped<Decode2Cfg>(&q, 1, B, 2, cbk, workspace, st);
        case 3: return run_grouped<Decode3Cfg>(&q, 1, B, 3, cbk, workspace, st);
        case 4: return run_grouped<DecodeCfg>(&q, 1, B, 4, cbk, workspace, st);
        // ternary: 2-bit fields, the level table {-c, 0, +c, 0}
        case CQ_TERNARY: return run_grouped<Decode2Cfg>(&q, 1, B, CQ_TERNARY, cbk, workspace, st);
        default: return CQ_ERR_UNSUPPORTED;
    }
}

}  // namespace cq


// ---------------------------------------------------------------------------------
// Q4_0 on the tensor cores: the activations are converted once to fp16 (workspace),
// then the persistent pipeline decodes each weight block once per tile of tokens.
// ---------------------------------------------------------------------------------
namespace cq {
namespace {

int64_t q40_padded_k(int64_t K) { return (K + 31) / 32 * 32; }

template <class C>
cq_status run_q40(const uint8_t* blocks, int64_t N, int64_t K, const float* X, int64_t M, float* Y,
                  void* workspace, cudaStream_t cs) {
    unsigned int* err = nullptr;
    cq_status st = host_setup(&err);
    if (st != CQ_OK) return st;
    const int64_t Kp = q40_padded_k(K);
    uint16_t* xh = static_cast<uint16_t*>(workspace);
    {
        const int64_t groups = M * (Kp / 8);
        int64_t grid = (groups + 255) / 256;
        const int64_t cap = (int64_t)sm_count() * 8;
        if (grid > cap) grid = cap;
        st = launch_pdl(q4_act_kernel, dim3((unsigned)grid), dim3(256), 0, cs, X, K, Kp, groups, xh);
        if (st != CQ_OK) return st;
    }
    static GemmParams prm;   // large; built on the host, passed by value to the launch
    std::lock_guard<std::mutex> lock(g_host_mu);
    memset(&prm, 0, sizeof(prm));
    st = make_act_map(&prm.tmap[0], xh, M, Kp, C::BT, true);
    if (st != CQ_OK) return st;
    GemmProblem& gp = prm.prob[0];
    gp.packed = blocks;
    gp.Y = Y;
    gp.N = (int)N;
    gp.K = (int)Kp;
    gp.act = 0;
    st = make_q40_map(&gp.pmap, blocks, N, Kp / 32);
    if (st != CQ_OK) return st;
    const int tiles_m = (int)((M + C::BT - 1) / C::BT);
    gp.tiles_n = (int)((N + kBO - 1) / kBO);
    gp.tile_begin = 0;
    choose_split<C>(gp, tiles_m, 4);   // Q4_0 splits on whole 256-column slabs
    if (gp.ksplit > 1) {
        const cudaError_t e = cudaMemsetAsync(Y, 0, (size_t)M * (size_t)N * sizeof(float), cs);
        if (e != cudaSuccess) { set_last_cuda_error((int)e); return CQ_ERR_CUDA; }
    }
    prm.nprob = 1;
    prm.M = (int)M;
    prm.tiles_m = tiles_m;
    prm.total_tiles = gp.tiles_per_split * gp.ksplit;
    prm.err = err;
    prm.timeout_ns = 2000000000ull;   // 2 s per wait
    const int grid = prm.total_tiles < sm_count() ? prm.total_tiles : sm_count();
    return launch_pdl(cq_gemm_kernel<C>, dim3(grid), dim3(C::THREADS), (size_t)kGemmSmem, cs, prm);
}

}  // namespace
}  // namespace cq

extern "C" size_t q4_0_gemm_workspace_bytes(int64_t M, int64_t K) {
    if (M < 1 || K < 1) return 0;
    return ((size_t)M * (size_t)cq::q40_padded_k(K) * 2u + 255u) & ~(size_t)255u;
}

extern "C" cq_status q4_0_gemm(const uint8_t* blocks, int64_t N, int64_t K, const float* X, int64_t M,
                               float* Y, void* workspace, size_t workspace_bytes, void* stream) {
    if (!blocks || !X || !Y || N < 1 || K < 1 || M < 1) return CQ_ERR_INVALID_ARG;
    if (M > (1 << 30) || N > (1 << 24) || K > (1 << 24) || M * N > ((int64_t)1 << 40))
        return CQ_ERR_UNSUPPORTED;
    // whole 256-k slabs: rows of a multiple of 8 blocks (also the 16-byte row stride the
    // tensor copies need)
    if ((cq::q40_padded_k(K) / 32) % 8 != 0) return CQ_ERR_UNSUPPORTED;
    if (!aligned16(blocks) || !aligned16(X) || !aligned16(Y)) return CQ_ERR_ALIGNMENT;
    if (!workspace || workspace_bytes < q4_0_gemm_workspace_bytes(M, K)) return CQ_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return CQ_ERR_ALIGNMENT;
    cudaStream_t cs = as_stream(stream);
    if (M <= 32) return run_q40<Q40NarrowCfg>(blocks, N, K, X, M, Y, workspace, cs);
    return run_q40<Q40WideCfg>(blocks, N, K, X, M, Y, workspace, cs);
}
