// Allocation-free variant of pkv_paged_attention_decode.
//
// Some callers cannot hand the library a device workspace: code that runs
// while a CUDA stream is being captured into a graph (cudaMalloc is not a
// capturable operation), plugins embedded in a host runtime that owns every
// device allocation and exposes no allocator, and serving loops whose memory
// was fully planned up front and must not call cudaMalloc / cudaFree (which
// can synchronise the device) on the decode path.  For them this entry point
// keeps the split-K partials in a fixed array that lives in the library
// itself: a file-scope __device__ array of PKV_STATIC_WORKSPACE_BYTES,
// present on every GPU that loads the library until the process exits.
//
// The computation is exactly pkv_paged_attention_decode's: this file only
// supplies the workspace pointer to the existing entry point.

#include <mutex>

#include "common.cuh"

namespace {

static __device__ __align__(256) unsigned char g_static_workspace[PKV_STATIC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_static_mu;
void* g_static_addr[kMaxDevices] = {nullptr};

// Device address of this device's array.  In host code the array's name is
// only a host-side stand-in, so the address is looked up with
// cudaGetSymbolAddress, once per device, with that device current.
int static_workspace(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PKV_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_static_mu);
    if (!g_static_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_workspace) != cudaSuccess || !p) return PKV_ERR_CUDA;
        g_static_addr[dev] = p;
    }
    *out = g_static_addr[dev];
    return PKV_OK;
}

}  // namespace

extern "C" int pkv_paged_attention_decode_static_ws(
    const void* q, const void* k_pool, const void* v_pool, const int32_t* block_tables,
    const int32_t* context_lens, int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
    int32_t head_dim, int32_t num_blocks, int32_t block_size, int32_t max_blocks, float scale,
    void* out, int32_t partition_size, int dtype, void* stream) {
    size_t need = 0;
    int st = pkv_decode_workspace_bytes(batch, num_q_heads, head_dim, max_blocks, block_size,
                                        partition_size, &need);
    if (st != PKV_OK) return st;
    if (need > static_cast<size_t>(PKV_STATIC_WORKSPACE_BYTES)) return PKV_ERR_WORKSPACE;
    void* ws = nullptr;
    size_t ws_bytes = 0;
    if (need > 0 && batch > 0) {
        if ((st = static_workspace(&ws)) != PKV_OK) return st;
        ws_bytes = PKV_STATIC_WORKSPACE_BYTES;
    }
    return pkv_paged_attention_decode(q, k_pool, v_pool, block_tables, context_lens, batch,
                                      num_q_heads, num_kv_heads, head_dim, num_blocks, block_size,
                                      max_blocks, scale, out, ws, ws_bytes, partition_size, dtype,
                                      stream);
}
