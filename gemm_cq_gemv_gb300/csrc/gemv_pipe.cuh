// Device pieces shared by the GEMV kernels (gemv.cu, gemv_dp.cu): mbarrier waits,
// 2-D tensor copies, the bump allocator of the shared window and the deterministic
// cross-warp reduction of a row tile.
//
// Every GEMV kernel is one persistent CTA per SM whose warps own fixed K-segments of a
// tile of kRows output rows, so each tile needs a cross-warp sum: a warp drops its
// per-row partials into one of kSlots shared slots and counts itself in with an atomic
// add on the slot's counter; the warp that arrives last adds the partials in warp order
// (deterministic), writes the rows and frees the slot.  A warp waits only when it runs
// kSlots tiles ahead of the slowest one.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"

namespace cq {
namespace pipe {

constexpr int kRows = 8;        // output rows per warp tile
constexpr int kSlots = 16;      // tiles whose reduction may be in flight

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

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
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
                     smem_u32(b)), "r"(bytes)
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
__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Bounded wait (2 s by default): on expiry raise the device error flag and give up (the
// result of the call is then undefined and cq_device_error() reports the timeout).
__device__ __forceinline__ void mbar_wait(uint64_t* b, uint32_t parity, unsigned int* err,
                                          unsigned long long timeout_ns = 2000000000ull) {
    if (mbar_try(b, parity)) return;
    const unsigned long long t0 = global_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try(b, parity)) return;
        if ((i & 255u) == 0u && global_ns() - t0 > timeout_ns) {
            atomicOr(err, 2u);
            return;
        }
    }
}

struct Reduce {
    // partial sums [kSlots][NW][TB][8]: the 32 floats of partial i / 32 start at
    // part + (i / 32) * pstride (pstride = 32 when the area is contiguous)
    float* part;
    int pstride;
    uint32_t* count;    // [kSlots] arrivals (cumulative)
    uint64_t* empty;    // [kSlots] completes when the slot's tile has been reduced
    __device__ __forceinline__ float& at(int i) const { return part[(i >> 5) * pstride + (i & 31)]; }
};

__device__ __forceinline__ uint32_t atomic_add_acq_rel_shared(uint32_t* a, uint32_t v) {
    uint32_t old;
    asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], %2;"
                 : "=r"(old)
                 : "r"(smem_u32(a)), "r"(v)
                 : "memory");
    return old;
}

// Stores this warp's row partials of tile number `it`; the last of the `nbusy` warps to
// arrive reduces the tile.  `fin(t, rr, sum)` receives the sum for token t of tile row rr.
template <int TB, int NW, typename Fin>
__device__ __forceinline__ void tile_reduce(const Reduce& rd, const float (&acc)[TB][kRows], int it,
                                            int w, int lane, int nsl, uint32_t nbusy, int tile_rows,
                                            int ntok, unsigned int* err, Fin fin) {
    const int slot = it % kSlots;
    const uint32_t ph = (uint32_t)((it / kSlots) & 1);
    float v[TB];
#pragma unroll
    for (int t = 0; t < TB; ++t) v[t] = reduce_rows8(acc[t], lane);
    mbar_wait(&rd.empty[slot], ph ^ 1u, err);
    if ((lane & 3) == 0) {
#pragma unroll
        for (int t = 0; t < TB; ++t)
            rd.at(((slot * NW + w) * TB + t) * kRows + ((lane >> 2) & 7)) = v[t];
    }
    __syncwarp();
    uint32_t old = 0;
    if (lane == 0) old = atomic_add_acq_rel_shared(&rd.count[slot], 1u);
    old = __shfl_sync(0xffffffffu, old, 0);
    if (old % nbusy == nbusy - 1u) {
        __syncwarp();
        for (int idx = lane; idx < TB * tile_rows; idx += 32) {
            const int t = idx / tile_rows, rr = idx % tile_rows;
            const int g = rr / kRows, r = rr % kRows;
            if (t < ntok) {
                float sum = 0.0f;
                for (int ss = 0; ss < nsl; ++ss)
                    sum += rd.at(((slot * NW + g * nsl + ss) * TB + t) * kRows + r);
                fin(t, rr, sum);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&rd.empty[slot]);
    }
}

// Stores this warp's row partials of its k-th row group; the last of the nsl warps of its
// warp set (the warps sharing the group, one per K-segment) to arrive adds them in warp
// order (deterministic) and hands fin(t, r, sum) the sums.  Each warp set has its own
// kSlots counters and barriers; a warp waits only when it runs kSlots groups ahead.
template <int TB, int NW, typename Fin>
__device__ __forceinline__ void group_reduce(const Reduce& rd, const float (&acc)[TB][kRows], int k, int w,
                                             int lane, int nsl, int rgi, int ntok, unsigned int* err, Fin fin) {
    const int ks = k % kSlots;
    const int sl = rgi * kSlots + ks;
    const uint32_t ph = (uint32_t)((k / kSlots) & 1);
    float v[TB];
#pragma unroll
    for (int t = 0; t < TB; ++t) v[t] = reduce_rows8(acc[t], lane);
    mbar_wait(&rd.empty[sl], ph ^ 1u, err);
    if ((lane & 3) == 0) {
#pragma unroll
        for (int t = 0; t < TB; ++t) rd.at(((ks * NW + w) * TB + t) * kRows + ((lane >> 2) & 7)) = v[t];
    }
    __syncwarp();
    uint32_t old = 0;
    if (lane == 0) old = atomic_add_acq_rel_shared(&rd.count[sl], 1u);
    old = __shfl_sync(0xffffffffu, old, 0);
    if (old % (uint32_t)nsl == (uint32_t)nsl - 1u) {
        __syncwarp();
        if (lane < TB * kRows) {
            const int t = lane / kRows, r = lane % kRows;
            if (t < ntok) {
                float sum = 0.0f;
                for (int ss = 0; ss < nsl; ++ss) sum += rd.at(((ks * NW + rgi * nsl + ss) * TB + t) * kRows + r);
                fin(t, r, sum);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&rd.empty[sl]);
    }
}

__device__ __forceinline__ void init_reduce(const Reduce& rd) {
    for (int s = 0; s < kSlots; ++s) {
        rd.count[s] = 0u;
        mbar_init(&rd.empty[s], 1);
    }
}

// bytes of the reduction area: partials, then the barriers (8-byte aligned), then counters
template <int NW>
__host__ __device__ constexpr size_t reduce_bytes(int tb) {
    return (size_t)kSlots * NW * tb * kRows * sizeof(float) + kSlots * sizeof(uint64_t) +
           kSlots * sizeof(uint32_t);
}

// the same area with kSlots counters and barriers for each of `nsets` warp sets
template <int NW>
__host__ __device__ constexpr size_t reduce_bytes_sets(int tb, int nsets) {
    return (size_t)kSlots * NW * tb * kRows * sizeof(float) + (size_t)nsets * kSlots * sizeof(uint64_t) +
           (size_t)nsets * kSlots * sizeof(uint32_t);
}

template <int NW>
__device__ __forceinline__ Reduce carve_reduce_sets(void* base, int tb, int nsets) {
    Reduce rd;
    rd.part = reinterpret_cast<float*>(base);
    rd.pstride = 32;
    rd.empty = reinterpret_cast<uint64_t*>(rd.part + kSlots * NW * tb * kRows);
    rd.count = reinterpret_cast<uint32_t*>(rd.empty + nsets * kSlots);
    return rd;
}

template <int NW>
__device__ __forceinline__ Reduce carve_reduce(void* base, int tb) {
    Reduce rd;
    rd.part = reinterpret_cast<float*>(base);
    rd.pstride = 32;
    rd.empty = reinterpret_cast<uint64_t*>(rd.part + kSlots * NW * tb * kRows);
    rd.count = reinterpret_cast<uint32_t*>(rd.empty + kSlots);
    return rd;
}

// 2-D tensor copy of one box (rows outside the tensor and columns past its end read as
// zero and still count toward the transaction bytes)
__device__ __forceinline__ void tma_box(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
// orders this thread's earlier shared-memory reads before later bulk copies into them
__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Bump allocator over (at most) two free ranges of the shared window; every thread runs
// it identically, so all agree on the layout.
struct SmemCarve {
    uint32_t a, a_end, b, b_end;
    bool ok;
    __device__ __forceinline__ uint32_t take(uint32_t size, uint32_t align) {
        const uint32_t pa = (a + align - 1) & ~(align - 1);
        if (pa + size <= a_end) { a = pa + size; return pa; }
        const uint32_t pb = (b + align - 1) & ~(align - 1);
        if (pb + size <= b_end) { b = pb + size; return pb; }
        ok = false;
        return b;
    }
};

// Host side (defined in gemv.cu).
// Cached device address of the GEMV unit's error word on the current device.
cq_status device_error_word(unsigned int** out);
// cuTensorMapEncodeTiled of a 2-D row-major array: `inner` elements per row of
// `row_bytes`, `rows` rows, box `box_inner` x `box_rows`, no swizzle, zero fill.
cq_status encode_map(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner,
                     uint64_t rows, uint64_t row_bytes, uint32_t box_inner, uint32_t box_rows);

}  // namespace pipe

// Batch-1 and batch-2 CQ GEMV of 4-bit rows on 16-bit integer codewords (gemv_fx.cu).
// Needs K % 1024 == 0, K <= 32768 and 16-byte aligned operands.  CQ_ERR_UNSUPPORTED
// when the level table is not finite or all zero (the caller then uses the fp32 kernel).
cq_status cq4_gemv_fx(const uint8_t* packed, const uint16_t* norms, int64_t N, int64_t K,
                      const cq_codebook* cbk, const int8_t* Xq, const float* scale, int64_t B,
                      float* Y, cudaStream_t st);

}  // namespace cq
