// Library-wide entry points of libcqgemv: status strings, error bookkeeping, version.
#include "common.cuh"

namespace cq {

namespace {
thread_local int g_last_cuda_error = 0;
int g_sm_count[64] = {0};
}  // namespace

void set_last_cuda_error(int code) { g_last_cuda_error = code; }

int sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
    if (g_sm_count[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
            n = 1;
        g_sm_count[dev] = n;
    }
    return g_sm_count[dev];
}

}  // namespace cq

extern "C" const char* cq_status_string(cq_status s) {
    switch (s) {
        case CQ_OK: return "CQ_OK";
        case CQ_ERR_INVALID_ARG: return "CQ_ERR_INVALID_ARG";
        case CQ_ERR_ALIGNMENT: return "CQ_ERR_ALIGNMENT";
        case CQ_ERR_UNSUPPORTED: return "CQ_ERR_UNSUPPORTED";
        case CQ_ERR_CUDA: return "CQ_ERR_CUDA";
        case CQ_ERR_DEVICE_TIMEOUT: return "CQ_ERR_DEVICE_TIMEOUT";
        case CQ_ERR_WORKSPACE: return "CQ_ERR_WORKSPACE";
    }
    return "CQ_ERR_UNKNOWN";
}

extern "C" int cq_last_cuda_error(void) { return cq::g_last_cuda_error; }

extern "C" int cq_abi_version(void) { return CQGEMV_ABI_VERSION; }

extern "C" cq_status cq_levels(int b, const cq_codebook* cbk, float* levels_out) {
    if (!levels_out || !cq::cq_code_valid(b)) return CQ_ERR_INVALID_ARG;
    if (!cbk && b != 1 && b != CQ_TERNARY) return CQ_ERR_INVALID_ARG;
    float lv[16];
    cq::cq_host_levels(lv, b, cbk);
    for (int t = 0; t < 16; ++t) levels_out[t] = lv[t];
    return CQ_OK;
}

extern "C" cq_status cq_device_error(void* stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) { cq::set_last_cuda_error((int)e); return CQ_ERR_CUDA; }
    unsigned int* words[2] = {cq::gemm_error_word(dev), cq::gemv_error_word(dev)};
    cudaStream_t cs = cq::as_stream(stream);
    bool raised = false;
    for (unsigned int* w : words) {
        if (!w) continue;   // no kernel of that unit launched on this device yet
        unsigned int host = 0;
        e = cudaMemcpyAsync(&host, w, sizeof(host), cudaMemcpyDeviceToHost, cs);
        if (e == cudaSuccess) e = cudaStreamSynchronize(cs);
        if (e != cudaSuccess) { cq::set_last_cuda_error((int)e); return CQ_ERR_CUDA; }
        if (host) {
            raised = true;
            const unsigned int zero = 0;
            e = cudaMemcpyAsync(w, &zero, sizeof(zero), cudaMemcpyHostToDevice, cs);
            if (e == cudaSuccess) e = cudaStreamSynchronize(cs);
            if (e != cudaSuccess) { cq::set_last_cuda_error((int)e); return CQ_ERR_CUDA; }
        }
    }
    return raised ? CQ_ERR_DEVICE_TIMEOUT : CQ_OK;
}

extern "C" cq_status cq_probe_bounded_wait(uint64_t timeout_ns, void* stream) {
    if (timeout_ns < 1000u || timeout_ns > 10000000000ull) return CQ_ERR_INVALID_ARG;
    cudaStream_t cs = cq::as_stream(stream);
    const cq_status s = cq::probe_gemm_wait(timeout_ns, cs);
    if (s != CQ_OK) return s;
    return cq::probe_gemv_wait(timeout_ns, cs);
}
