// Per-device status word: kernels OR PKV_STATUS_* bits into it when a
// data-dependent index (table entry, slot, context length, copy pair, sink
// row) is out of range; the access itself is skipped.  pkv_device_status
// reads and clears it.

#include <mutex>

#include "common.cuh"

namespace {

__device__ int g_status_word;

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int* g_addr[kMaxDevices] = {nullptr};

}  // namespace

namespace pkv {

int* status_word() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
        g_addr[dev] = static_cast<int*>(p);
    }
    return g_addr[dev];
}

}  // namespace pkv

extern "C" int pkv_device_status(int32_t* status, void* stream) {
    if (!status) return PKV_ERR_INVALID_ARG;
    int* w = pkv::status_word();
    if (!w) return PKV_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int host = 0;
    if (cudaMemcpyAsync(&host, w, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return PKV_ERR_CUDA;
    if (cudaMemsetAsync(w, 0, sizeof(int), s) != cudaSuccess) return PKV_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return PKV_ERR_CUDA;
    *status = host;
    return host ? PKV_ERR_DEVICE_BOUNDS : PKV_OK;
}
