// Multi-query paged attention on the 5th-generation tensor cores (tcgen05 +
// TMA), for long query spans: chunked-prefill slices (prefill_tc.cu).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace pkv {

// Rows (query tokens x G) per (sequence, KV head) above which a call takes
// the tensor-core kernel.
constexpr int kPrefillTcMinRows = 64;

// Whether the tensor-core kernel serves this shape: head dim 128, a GQA
// group of 1, 2, 4 or 8, more than kPrefillTcMinRows rows.
bool prefill_tc_applies(int head_dim, int G, int64_t rows);

// Launches it (arguments as pkv_paged_attention_multi_query, already
// checked); PKV_ERR_CUDA if a tensor map cannot be made or the launch fails.
int launch_prefill_tc(const void* q, const int32_t* q_start, const void* k_pool, const void* v_pool,
                      const int32_t* tables, const int32_t* ctx_lens, int batch, int hq, int hkv, int num_blocks,
                      int max_blocks, int max_q_len, float scale, void* out, int* status, bool bf16,
                      cudaStream_t st);

}  // namespace pkv
