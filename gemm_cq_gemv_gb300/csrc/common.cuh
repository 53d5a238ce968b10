// Shared device/host helpers of libcqgemv (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "cqgemv.h"

namespace cq {

constexpr int kGroup = 128;

// Remembers the last CUDA error code per host thread (cq_last_cuda_error).
void set_last_cuda_error(int code);

inline cq_status check_launch() {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_last_cuda_error((int)e);
        return CQ_ERR_CUDA;
    }
    return CQ_OK;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// CQ codes: b = 1..4 index bits (2^b Lloyd-Max levels), or CQ_TERNARY = 5, the fixed
// three-level codebook {-c, 0, +c} of the Needle mmap page whose indices 0, 1, 2 sit in
// 2-bit fields.
inline bool cq_code_valid(int b) { return (b >= 1 && b <= 4) || b == CQ_TERNARY; }
// Bits of one packed index field (a group holds 16 * field bytes).
inline int cq_field_bits(int b) { return b == CQ_TERNARY ? 2 : b; }

// The level table a kernel reads for code b (ascending; unused entries 0).
//  b = 1: the fixed +-sqrt(2/pi) (Needle mmap page: mean of |N(0,1)|).
//  b = 5: the fixed {-c, 0, +c}.  The page gives no c; c is the three-level Lloyd-Max
//         level of N(0,1), the root of c = phi(c/2) / (1 - Phi(c/2)) (thresholds at
//         +-c/2, the outer level the mean of the tail beyond them).  Entry 3 of the 2-bit
//         field never occurs in an encoding and reads as 0.
//  b = 2..4: cb2 | cb3 | cb4 of the caller's table.
inline void cq_host_levels(float (&lv)[16], int b, const cq_codebook* cbk) {
    for (int t = 0; t < 16; ++t) lv[t] = 0.0f;
    if (b == 1) {
        const float c = 0.797884560802865355879892119868763737f;   // sqrt(2/pi)
        lv[0] = -c; lv[1] = c;
        return;
    }
    if (b == CQ_TERNARY) {
        const float c = 1.224006361924961521136180602132438972f;
        lv[0] = -c; lv[1] = 0.0f; lv[2] = c;
        return;
    }
    const int off = (b == 2) ? 0 : (b == 3) ? 4 : 12;
    for (int t = 0; t < (1 << b); ++t) lv[t] = cbk->cb[off + t];
}
// Number of levels of code b.
inline int cq_num_levels(int b) { return b == CQ_TERNARY ? 3 : 1 << b; }

inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

// Programmatic dependent launch.  A kernel launched with launch_pdl may start while the
// previous kernel of the stream is still finishing; it calls pdl_wait() before its first
// global-memory access (which then sees everything the previous kernel wrote) and
// pdl_trigger() once all its blocks are resident, so the next launch can begin early.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;"); }

template <typename... Params, typename... Args>
cq_status launch_pdl(void (*kern)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                     Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
    if (e != cudaSuccess) {
        set_last_cuda_error((int)e);
        return CQ_ERR_CUDA;
    }
    return check_launch();
}

// Number of SMs of the current device (cached per device).
int sm_count();

// Device error words raised by bounded waits (one file-scope __device__ word per
// translation unit); each returns the cached device address for `dev`, or nullptr if
// no kernel of that unit has been set up on it yet.
unsigned int* gemm_error_word(int dev);
unsigned int* gemv_error_word(int dev);

// Failure-detection probes (one per unit): a one-thread kernel whose bounded wait on a
// barrier phase that nothing completes gives up after `timeout_ns` and raises the unit's
// error word.
cq_status probe_gemm_wait(unsigned long long timeout_ns, cudaStream_t st);
cq_status probe_gemv_wait(unsigned long long timeout_ns, cudaStream_t st);

// float64 -> IEEE binary16 bits, one round-to-nearest-even step (ties to even),
// written from the binary16 definition: 1 sign bit, 5 exponent bits (bias 15),
// 10 fraction bits, subnormals with unit 2^-24, overflow to infinity.
__device__ __forceinline__ uint16_t f64_to_f16_bits_rne(double x) {
    unsigned long long u = (unsigned long long)__double_as_longlong(x);
    uint32_t sign = (uint32_t)(u >> 48) & 0x8000u;
    u &= 0x7FFFFFFFFFFFFFFFull;
    uint32_t ebits = (uint32_t)(u >> 52);
    if (ebits == 0x7FF) {  // inf / nan
        return (uint16_t)(sign | 0x7C00u | ((u & 0xFFFFFFFFFFFFFull) ? 0x200u : 0u));
    }
    if (ebits == 0) return (uint16_t)sign;  // float64 zero / subnormal -> signed zero
    int e = (int)ebits - 1023;
    unsigned long long m = (u & 0xFFFFFFFFFFFFFull) | (1ull << 52);  // 53-bit significand
    if (e > 15) return (uint16_t)(sign | 0x7C00u);
    if (e >= -14) {
        unsigned long long hm = m >> 42;                 // 11 bits incl. the leading one
        unsigned long long rem = m & ((1ull << 42) - 1);
        const unsigned long long half = 1ull << 41;
        if (rem > half || (rem == half && (hm & 1ull))) hm++;
        uint32_t eh = (uint32_t)(e + 15);
        if (hm == 2048ull) { hm = 1024ull; eh++; }
        if (eh >= 31u) return (uint16_t)(sign | 0x7C00u);
        return (uint16_t)(sign | (eh << 10) | (uint32_t)(hm & 0x3FFull));
    }
    // subnormal binary16: value / 2^-24 = m * 2^(e - 28)
    int shift = 28 - e;                                   // >= 43
    if (shift >= 64) return (uint16_t)sign;
    unsigned long long q = m >> shift;
    unsigned long long rem = m & ((1ull << shift) - 1);
    unsigned long long half = 1ull << (shift - 1);
    if (rem > half || (rem == half && (q & 1ull))) q++;
    return (uint16_t)(sign | (uint32_t)q);               // q == 1024 is the smallest normal
}

// Batched cq_gemv (1- to 4-bit indices) through the tensor-core pipeline of gemm.cu: fp16
// operands, fp32 output; workspace >= B * K * 2 + 256 bytes, 16-byte aligned.
cq_status gemv_tensor(const uint8_t* packed, const uint16_t* norms, int64_t N, int64_t K, int b,
                      const cq_codebook* cbk, const int8_t* Xq, const float* scale, int64_t B,
                      float* Y, void* workspace, cudaStream_t st);

// IEEE binary16 bits -> float32 (exact).
__device__ __forceinline__ float f16_bits_to_f32(uint16_t h) {
    return __half2float(__ushort_as_half(h));
}

}  // namespace cq
