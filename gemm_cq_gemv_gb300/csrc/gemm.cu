// Prefill GEMM for CQ-W4A8 weights on the 5th-generation tensor cores (A6).
//
// "14MB 装下 45M 参数…", §三: prefill is a GEMM over the same pre-transposed [out, in]
// rows the decode GEMV streams; §一: w_group = (cb[idx] * norm / sqrt(128)) @ H.  With
// xr = Hu @ q (the rotated int8 activations, exact integers) the product is
//   Y[t][o] = s_t / 128 * sum_k xr[t][k] * cb[idx[o][k]] * norm[o][k / 128]
// and both factors of the contraction are fed to tcgen05.mma as bf16:
//   A = bf16(xr)                [M tokens][K]      - rotated once per call, TMA-loaded
//   B = bf16(cb[idx] * norm)    [N out-rows][K]    - dequantised in shared memory
// with fp32 accumulation in tensor memory and a bf16 epilogue.
//
// One CTA per SM (persistent), tile = 256 tokens x 128 out-rows, K in chunks of 64 (one
// 128-byte swizzle atom of bf16), 4 stages; the two fp32 accumulators of a tile (one per
// 128-token half) are double-buffered in tensor memory so the epilogue of a tile runs
// under the main loop of the next.
// Warp roles:
//   warp 0      TMA producer: per stage the two 128-token A tiles and the packed 4-bit
//               weight tile (128 rows x 32 bytes)
//   warp 1      MMA issuer (one thread): 2 x 4 tcgen05.mma (M=128, N=128, K=16) per stage
//   warps 2-9   epilogue: tcgen05.ld of the two accumulators (two warps per TMEM lane
//               quarter, 64 columns each), scale, bf16, store
//   warps 10-17 dequant: packed tile (shared) -> bf16 B tile in the SWIZZLE_128B layout
// Every mbarrier wait is bounded (globaltimer); on expiry the CTA raises a device error
// flag, stops issuing work, frees its tensor memory and returns.

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <mutex>

#include "common.cuh"

namespace cq {
namespace {

constexpr int kBM = 256;                 // tokens per tile (two M=128 MMAs)
constexpr int kBN = 128;                 // out-rows per tile (MMA N)
constexpr int kBK = 64;                  // K per stage (128 bytes of bf16)
constexpr int kStages = 4;
constexpr int kThreadsGemm = 576;        // 18 warps
constexpr int kEpiWarp0 = 2;             // warps 2..9: two per TMEM lane quarter
constexpr int kEpiWarps = 8;
constexpr int kDequantWarp0 = kEpiWarp0 + kEpiWarps;
constexpr int kDequantThreads = 256;     // warps 10..17
constexpr int kATileBytes = 128 * kBK * 2;           // 16 KB
constexpr int kBTileBytes = kBN * kBK * 2;           // 16 KB
constexpr int kPTileBytes = kBN * kBK / 2;           // 4 KB of packed nibbles
constexpr int kStageBytes = 2 * kATileBytes + kBTileBytes + kPTileBytes;
constexpr int kTmemCols = 512;                       // 2 buffers x 2 halves x 128 columns
constexpr int kMaxProblems = 120;
constexpr int kMaxActs = 8;

struct GemmProblem {
    CUtensorMap pmap;        // packed bytes as [N][K/2] uint8, box 32 x 128
    const uint8_t* packed;   // [N][K/128][64]
    const uint16_t* norms;   // [N][K/128]
    const float* scale;      // [M]
    __nv_bfloat16* Y;        // [M][N]
    int N, K;
    int act;                 // index of the activation tensor map
    int tiles_n;
    int tile_begin;          // first global tile index of this problem
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
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(smem_u32(b)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait: false when the deadline passed or another thread already aborted.
__device__ __forceinline__ bool mbar_wait(uint64_t* b, uint32_t parity, volatile int* abort_flag,
                                          const GemmParams& p) {
    if (mbar_try(b, parity)) return true;
    const unsigned long long t0 = global_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try(b, parity)) return true;
        if ((i & 255u) == 0u) {
            if (*abort_flag) return false;
            if (global_ns() - t0 > p.timeout_ns) {
                *abort_flag = 1;
                atomicOr(p.err, 1u);
                return false;
            }
        }
    }
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

// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, both K-major.
__host__ __device__ constexpr uint32_t idesc_bf16(int m, int n) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) |
           ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
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
__device__ __forceinline__ void tmem_ld32_async(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
        "%28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// scale the first `valid` (0, 16 or 32) of 32 fp32 accumulator columns, round to bf16
// and store them contiguously
__device__ __forceinline__ void store_row32(__nv_bfloat16* dst, const uint32_t (&r)[32], float sc,
                                            int valid) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        if (8 * q >= valid) break;
        uint4 o;
        uint32_t* w = &o.x;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            __nv_bfloat162 v = __floats2bfloat162_rn(__uint_as_float(r[8 * q + 2 * j]) * sc,
                                                     __uint_as_float(r[8 * q + 2 * j + 1]) * sc);
            w[j] = *reinterpret_cast<uint32_t*>(&v);
        }
        *reinterpret_cast<uint4*>(dst + 8 * q) = o;
    }
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
// xr = bf16(Hu @ q) per 128-group; one warp per (token, group).  The fp32 butterfly is
// exact (integers below 2^24); the single rounding is the bf16 conversion.
// ---------------------------------------------------------------------------------
__global__ void __launch_bounds__(256)
rotate_act_bf16_kernel(const int8_t* __restrict__ Xq, int64_t groups, __nv_bfloat16* __restrict__ out) {
    const int lane = threadIdx.x & 31;
    const int64_t warp = ((int64_t)blockIdx.x * 256 + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * 256) >> 5;
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
        __nv_bfloat162 lo = __floats2bfloat162_rn(v0, v1);
        __nv_bfloat162 hi = __floats2bfloat162_rn(v2, v3);
        uint2 pk;
        pk.x = *reinterpret_cast<uint32_t*>(&lo);
        pk.y = *reinterpret_cast<uint32_t*>(&hi);
        *reinterpret_cast<uint2*>(out + gi * kGroup + 4 * lane) = pk;
    }
}

// ---------------------------------------------------------------------------------
// The persistent tcgen05 GEMM.
// ---------------------------------------------------------------------------------
struct TileRef {
    int prob, mt, nt;
};

__device__ __forceinline__ TileRef tile_ref(const GemmParams& p, int tile) {
    TileRef t;
    t.prob = find_problem(p, tile);
    const int local = tile - p.prob[t.prob].tile_begin;
    t.mt = local % p.tiles_m;
    t.nt = local / p.tiles_m;
    return t;
}

// norm (as fp32) of row `o` for K-chunk `kc`, 0 for rows past N
__device__ __forceinline__ float load_norm(const GemmProblem& pr, int o, int kc) {
    if (o >= pr.N) return 0.0f;
    const int G = pr.K / kGroup;
    return f16_bits_to_f32(__ldg(pr.norms + (int64_t)o * G + (kc * kBK) / kGroup));
}

__global__ void __launch_bounds__(kThreadsGemm, 1) cq_gemm_kernel(const __grid_constant__ GemmParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~(uintptr_t)1023);
    // stage s: [A half 0 | A half 1 | B (bf16, swizzled) | P (packed, 32 B per row)]
    uint8_t* stage_base = smem;
    float* lut = reinterpret_cast<float*>(smem + kStages * kStageBytes);        // [16][32]
    uint64_t* bars = reinterpret_cast<uint64_t*>(lut + 16 * 32);
    uint64_t* full_a = bars;                      // TMA: A tiles + packed tile landed
    uint64_t* full_b = bars + kStages;            // dequant: B tile written
    uint64_t* empty = bars + 2 * kStages;         // MMA: stage consumed
    uint64_t* acc_full = bars + 3 * kStages;      // [2] accumulator buffer ready
    uint64_t* acc_empty = acc_full + 2;           // [2] accumulator buffer drained
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 2);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    for (int i = tid; i < 16 * 32; i += kThreadsGemm) {
        const int t = i >> 5;
        float v = 0.0f;
#pragma unroll
        for (int u = 0; u < 16; ++u) v = (u == t) ? p.lv[u] : v;
        lut[i] = v;
    }
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full_a[s], 1);
            mbar_init(&full_b[s], kDequantThreads / 32);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], kEpiWarps);
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
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ------------------------------ TMA producer ------------------------------
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < p.total_tiles; tile += gridDim.x) {
                const TileRef tr = tile_ref(p, tile);
                const GemmProblem& pr = p.prob[tr.prob];
                const CUtensorMap* amap = &p.tmap[pr.act];
                for (int kc = 0; kc < pr.K / kBK; ++kc) {
                    if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag, p)) { ok = false; break; }
                    uint8_t* st = stage_base + s * kStageBytes;
                    mbar_arrive_tx(&full_a[s], 2 * kATileBytes + kPTileBytes);
                    tma_load_2d(st, amap, kc * kBK, tr.mt * kBM, &full_a[s]);
                    tma_load_2d(st + kATileBytes, amap, kc * kBK, tr.mt * kBM + 128, &full_a[s]);
                    tma_load_2d(st + 2 * kATileBytes + kBTileBytes, &pr.pmap, kc * (kBK / 2),
                                tr.nt * kBN, &full_a[s]);
                    if (++s == kStages) { s = 0; ph ^= 1u; }
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------ MMA issuer --------------------------------
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16(128, kBN);
            int s = 0;
            uint32_t ph = 0;
            int it = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < p.total_tiles; tile += gridDim.x, ++it) {
                const GemmProblem& pr = p.prob[find_problem(p, tile)];
                const int buf = it & 1;
                const uint32_t aph = (uint32_t)((it >> 1) & 1);
                if (!mbar_wait(&acc_empty[buf], aph ^ 1u, abort_flag, p)) break;
                tc_fence_after();
                const uint32_t d0 = tmem_base + (uint32_t)(buf * 2 * kBN);
                const int nk = pr.K / kBK;
                for (int kc = 0; kc < nk; ++kc) {
                    if (!mbar_wait(&full_a[s], ph, abort_flag, p) ||
                        !mbar_wait(&full_b[s], ph, abort_flag, p)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t st = smem_u32(stage_base + s * kStageBytes);
                    const uint64_t bdesc0 = smem_desc_sw128(st + 2 * kATileBytes);
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const uint64_t adesc0 = smem_desc_sw128(st + h * kATileBytes);
#pragma unroll
                        for (int kk = 0; kk < kBK / 16; ++kk) {
                            // +32 bytes along K inside the swizzle atom = +2 in the
                            // 16-byte-unit start address field
                            umma_bf16(d0 + (uint32_t)(h * kBN), adesc0 + 2u * kk, bdesc0 + 2u * kk,
                                      idesc, (kc > 0 || kk > 0) ? 1u : 0u);
                        }
                    }
                    umma_commit(&empty[s]);
                    if (++s == kStages) { s = 0; ph ^= 1u; }
                }
                if (!ok) break;
                umma_commit(&acc_full[buf]);
            }
        }
        __syncwarp();
    } else if (warp < kDequantWarp0) {
        // ------------------------------ epilogue ----------------------------------
        // warp -> TMEM lane quarter q (tokens 32q..32q+31 of each half) and a 64-column
        // half ch of the tile; four 32-column loads per tile, each issued before the
        // previous one is converted and stored
        const int q = warp & 3;
        const int ch = (warp - kEpiWarp0) >> 2;
        int it = 0;
        for (int tile = blockIdx.x; tile < p.total_tiles; tile += gridDim.x, ++it) {
            const TileRef tr = tile_ref(p, tile);
            const GemmProblem& pr = p.prob[tr.prob];
            const int buf = it & 1;
            if (!mbar_wait(&acc_full[buf], (uint32_t)((it >> 1) & 1), abort_flag, p)) break;
            tc_fence_after();
            const uint32_t lane_base = tmem_base + ((uint32_t)(q * 32) << 16) +
                                       (uint32_t)(buf * 2 * kBN + ch * 64);
            const int tok0 = tr.mt * kBM + q * 32 + lane;
            const int tok1 = tok0 + 128;
            const float sc0 = (tok0 < p.M) ? __ldg(pr.scale + tok0) * (1.0f / 128.0f) : 0.0f;
            const float sc1 = (tok1 < p.M) ? __ldg(pr.scale + tok1) * (1.0f / 128.0f) : 0.0f;
            const int col = tr.nt * kBN + ch * 64;
            __nv_bfloat16* y0 = pr.Y + (int64_t)tok0 * pr.N + col;
            __nv_bfloat16* y1 = pr.Y + (int64_t)tok1 * pr.N + col;
            // valid columns of each 32-column piece (N is a multiple of 16)
            const int v0 = min(32, max(0, pr.N - col)), v1 = min(32, max(0, pr.N - col - 32));
            uint32_t ra[32], rb[32];
            tmem_ld32_async(lane_base, ra);                         // half 0, cols 0..31
            tmem_wait_ld();
            tmem_ld32_async(lane_base + 32, rb);                    // half 0, cols 32..63
            if (tok0 < p.M) store_row32(y0, ra, sc0, v0);
            tmem_wait_ld();
            tmem_ld32_async(lane_base + kBN, ra);                   // half 1, cols 0..31
            if (tok0 < p.M) store_row32(y0 + 32, rb, sc0, v1);
            tmem_wait_ld();
            tmem_ld32_async(lane_base + kBN + 32, rb);              // half 1, cols 32..63
            if (tok1 < p.M) store_row32(y1, ra, sc1, v0);
            tmem_wait_ld();
            if (tok1 < p.M) store_row32(y1 + 32, rb, sc1, v1);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[buf]);
        }
    } else {
        // ------------------------------ dequant -----------------------------------
        // thread dt owns row r = dt / 2 and k-half hf = dt % 2 of every B tile: 32 nibbles
        // (16 bytes of the staged packed tile) -> four 16-byte chunks of the swizzled tile
        const int dt = tid - kDequantWarp0 * 32;    // 0..255
        const int r = dt >> 1, hf = dt & 1;
        const float* mylut = lut + lane;
        int s = 0;
        uint32_t ph = 0;
        bool ok = true;
        int tile = blockIdx.x;
        float nrm = 0.0f;
        if (tile < p.total_tiles) {
            const TileRef tr = tile_ref(p, tile);
            nrm = load_norm(p.prob[tr.prob], tr.nt * kBN + r, 0);
        }
        for (; ok && tile < p.total_tiles; tile += gridDim.x) {
            const TileRef tr = tile_ref(p, tile);
            const GemmProblem& pr = p.prob[tr.prob];
            const int nk = pr.K / kBK;
            for (int kc = 0; kc < nk; ++kc) {
                // prefetch the norm of the next chunk (or of the next tile's first chunk)
                float nrm_next = 0.0f;
                if (kc + 1 < nk) {
                    nrm_next = load_norm(pr, tr.nt * kBN + r, kc + 1);
                } else if (tile + (int)gridDim.x < p.total_tiles) {
                    const TileRef tn = tile_ref(p, tile + gridDim.x);
                    nrm_next = load_norm(p.prob[tn.prob], tn.nt * kBN + r, 0);
                }
                if (!mbar_wait(&full_a[s], ph, abort_flag, p)) { ok = false; break; }
                uint8_t* st = stage_base + s * kStageBytes;
                uint8_t* bt = st + 2 * kATileBytes;
                const uint4 w = *reinterpret_cast<const uint4*>(st + 2 * kATileBytes + kBTileBytes +
                                                                r * 32 + hf * 16);
                const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {      // 8 k values -> one 16-byte chunk
                    uint32_t pk[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const uint32_t i0 = (wv[j] >> (8 * e)) & 15u;
                        const uint32_t i1 = (wv[j] >> (8 * e + 4)) & 15u;
                        __nv_bfloat162 v = __floats2bfloat162_rn(mylut[i0 << 5] * nrm,
                                                                 mylut[i1 << 5] * nrm);
                        pk[e] = *reinterpret_cast<uint32_t*>(&v);
                    }
                    const int c = hf * 4 + j;
                    *reinterpret_cast<uint4*>(bt + r * 128 + ((c ^ (r & 7)) << 4)) =
                        make_uint4(pk[0], pk[1], pk[2], pk[3]);
                }
                // make the generic-proxy writes visible to the tensor cores, then arrive
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) mbar_arrive(&full_b[s]);
                if (++s == kStages) { s = 0; ph ^= 1u; }
                nrm = nrm_next;
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
bool g_attr_done[64] = {false};

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
    if (!g_attr_done[dev]) {
        const size_t smem = (size_t)kStages * kStageBytes + 16 * 32 * 4 + 256 + 1024;  // + align slack
        e = cudaFuncSetAttribute(cq_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) { set_last_cuda_error((int)e); return CQ_ERR_CUDA; }
        g_attr_done[dev] = true;
    }
    *err = g_err_ptr[dev];
    return CQ_OK;
}

cq_status make_packed_map(CUtensorMap* map, const void* base, int64_t N, int64_t K) {
    cuuint64_t dims[2] = {(cuuint64_t)(K / 2), (cuuint64_t)N};
    cuuint64_t strides[1] = {(cuuint64_t)(K / 2)};
    cuuint32_t box[2] = {(cuuint32_t)(kBK / 2), (cuuint32_t)kBN};
    cuuint32_t estr[2] = {1u, 1u};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) { set_last_cuda_error((int)r); return CQ_ERR_CUDA; }
    return CQ_OK;
}

cq_status make_act_map(CUtensorMap* map, const void* base, int64_t M, int64_t K) {
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
    cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    cuuint32_t box[2] = {(cuuint32_t)kBK, 128u};
    cuuint32_t estr[2] = {1u, 1u};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) { set_last_cuda_error((int)r); return CQ_ERR_CUDA; }
    return CQ_OK;
}

void fill_levels(float (&lv)[16], int b, const cq_codebook* cbk) {
    for (int t = 0; t < 16; ++t) lv[t] = 0.0f;
    const int off = (b == 2) ? 0 : (b == 3) ? 4 : 12;
    for (int t = 0; t < (1 << b); ++t) lv[t] = cbk->cb[off + t];
}

}  // namespace

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

extern "C" cq_status cq_gemm_grouped(const cq_gemm_problem* probs, int count, int64_t M, int g,
                                     int b, const cq_codebook* cbk, void* workspace,
                                     size_t workspace_bytes, void* stream) {
    if (!probs || count < 1 || !cbk || M < 1 || M > (1 << 30)) return CQ_ERR_INVALID_ARG;
    if (g != kGroup || b < 1 || b > 4) return CQ_ERR_INVALID_ARG;
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

    unsigned int* err = nullptr;
    cq_status st = host_setup(&err);
    if (st != CQ_OK) return st;
    cudaStream_t cs = as_stream(stream);

    // distinct activations -> rotated bf16 copies in the workspace
    if (count > 1024) return CQ_ERR_UNSUPPORTED;
    const int8_t* act_src[1024];
    const void* act_dst[1024];
    int64_t act_K[1024];
    int act_of[1024];
    int nact = 0;
    size_t off = 0;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    for (int i = 0; i < count; ++i) {
        int a = -1;
        for (int j = 0; j < nact; ++j)
            if (act_src[j] == probs[i].Xq) { a = j; break; }
        if (a < 0) {
            a = nact++;
            act_src[a] = probs[i].Xq;
            act_dst[a] = ws + off;
            act_K[a] = probs[i].K;
            const int64_t groups = M * (probs[i].K / kGroup);
            int64_t grid = (groups + 7) / 8;
            const int64_t cap = (int64_t)sm_count() * 16;
            if (grid > cap) grid = cap;
            rotate_act_bf16_kernel<<<(unsigned)grid, 256, 0, cs>>>(
                probs[i].Xq, groups, reinterpret_cast<__nv_bfloat16*>(ws + off));
            st = check_launch();
            if (st != CQ_OK) return st;
            off += ((size_t)M * (size_t)probs[i].K * 2u + 255u) & ~(size_t)255u;
        }
        act_of[i] = a;
    }

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
        const int tiles_m = (int)((M + kBM - 1) / kBM);
        while (i0 < count && np < kMaxProblems) {
            const int pi = order[i0];
            const int a = act_of[pi];
            if (map_of_act[a] < 0) {
                if (nmaps == kMaxActs) break;
                st = make_act_map(&prm.tmap[nmaps], act_dst[a], M, act_K[a]);
                if (st != CQ_OK) return st;
                map_of_act[a] = nmaps++;
            }
            const cq_gemm_problem& q = probs[pi];
            GemmProblem& gp = prm.prob[np++];
            gp.packed = q.packed; gp.norms = q.norms; gp.scale = q.scale;
            gp.Y = reinterpret_cast<__nv_bfloat16*>(q.Y);
            gp.N = (int)q.N; gp.K = (int)q.K; gp.act = map_of_act[a];
            st = make_packed_map(&gp.pmap, q.packed, q.N, q.K);
            if (st != CQ_OK) return st;
            gp.tiles_n = (int)((q.N + kBN - 1) / kBN);
            gp.tile_begin = tiles;
            tiles += gp.tiles_n * tiles_m;
            ++i0;
        }
        prm.nprob = np;
        prm.M = (int)M;
        prm.tiles_m = tiles_m;
        prm.total_tiles = tiles;
        fill_levels(prm.lv, b, cbk);
        prm.err = err;
        prm.timeout_ns = 2000000000ull;   // 2 s per wait
        const size_t smem = (size_t)kStages * kStageBytes + 16 * 32 * 4 + 256 + 1024;  // + align slack
        const int grid = tiles < sm_count() ? tiles : sm_count();
        cq_gemm_kernel<<<grid, kThreadsGemm, smem, cs>>>(prm);
        st = check_launch();
        if (st != CQ_OK) return st;
    }
    return CQ_OK;
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

