// KV-append scatter (plain and quantised) and the copy-on-write block copy.
//
// * pkv_kv_append: each decode step writes one new K/V vector per sequence
//   into the cache ("The 8GB VRAM Breakthrough", §1), at the slot the block
//   table reserved (§3).  A pure byte scatter, 16-byte vectors.
// * pkv_kv_append_quant: the fused quantiser on the write path (§5 flowchart,
//   "Fused Triton Quantizer (Per-Group Asymmetric INT4 / FP8)"), with the
//   first n_sink tokens also kept in 16-bit (§4 "Sink Window").  One warp per
//   (token, KV head, K|V) row; every arithmetic step is an IEEE binary32
//   operation with explicit rounding (__fsub_rn / __fdiv_rn / __fadd_rn /
//   rintf / __float2half_rn), never contracted, so the codes are bit-exact
//   with a binary32 reference.
// * pkv_copy_blocks: copy-on-write clone of whole physical blocks (§3 "Copy-on-
//   Write (CoW) Prefix Sharing").

#include "common.cuh"

namespace pkv {
namespace {

__global__ void kv_append_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                                 const int64_t* __restrict__ slots, int64_t total, int hkv,
                                 int cpr, int block_size, int64_t num_slots,
                                 uint4* __restrict__ kp, uint4* __restrict__ vp,
                                 int* __restrict__ status) {
    // a grid launched behind this one with programmatic serialization may be
    // scheduled now (it waits for this grid to complete before reading)
    asm volatile("griddepcontrol.launch_dependents;");
    const int64_t per_tok = static_cast<int64_t>(hkv) * cpr;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t t = i / per_tok;
        const int64_t rem = i - t * per_tok;
        const int64_t slot = slots[t];
        if (slot < 0) continue;
        if (slot >= num_slots) {
            if (rem == 0) atomicOr(status, PKV_STATUS_BAD_SLOT);
            continue;
        }
        const int h = static_cast<int>(rem / cpr);
        const int ch = static_cast<int>(rem - static_cast<int64_t>(h) * cpr);
        const int64_t blk = slot / block_size, off = slot - blk * block_size;
        const int64_t dst = ((blk * hkv + h) * block_size + off) * cpr + ch;
        kp[dst] = k[i];
        vp[dst] = v[i];
    }
}

// fp16 rounding that saturates to +-65504 instead of overflowing to inf.
__device__ __forceinline__ __half f16_sat(float x) {
    __half h = __float2half_rn(x);
    if (__hisinf(h)) h = __float2half_rn(x > 0.f ? 65504.f : -65504.f);
    return h;
}

template <typename T, int EPL>
__device__ __forceinline__ void load_row(const T* p, float (&x)[EPL]) {
    // EPL consecutive 16-bit values
    if constexpr (EPL == 2) {
        uint32_t w = *reinterpret_cast<const uint32_t*>(p);
        const T* e = reinterpret_cast<const T*>(&w);
        x[0] = Half16<T>::to_float(e[0]);
        x[1] = Half16<T>::to_float(e[1]);
    } else if constexpr (EPL == 4) {
        uint2 w = *reinterpret_cast<const uint2*>(p);
        const T* e = reinterpret_cast<const T*>(&w);
#pragma unroll
        for (int i = 0; i < 4; ++i) x[i] = Half16<T>::to_float(e[i]);
    } else {
        uint4 w = *reinterpret_cast<const uint4*>(p);
        const T* e = reinterpret_cast<const T*>(&w);
#pragma unroll
        for (int i = 0; i < 8; ++i) x[i] = Half16<T>::to_float(e[i]);
    }
}

template <typename T, int EPL>
__device__ __forceinline__ void copy_row(const T* src, T* dst) {
    if constexpr (EPL == 2) {
        *reinterpret_cast<uint32_t*>(dst) = *reinterpret_cast<const uint32_t*>(src);
    } else if constexpr (EPL == 4) {
        *reinterpret_cast<uint2*>(dst) = *reinterpret_cast<const uint2*>(src);
    } else {
        *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(src);
    }
}

struct QuantArgs {
    const void* k;
    const void* v;
    const int64_t* slots;
    const int32_t* positions;
    const int32_t* seq_idx;
    int T, hkv, D, block_size, group_size, n_sink, sink_rows;
    int64_t num_slots;
    uint8_t* codes[2];
    __half* scale[2];
    __half* zero[2];
    void* sink[2];
    void* win[2];        // 16-bit window rings [sink_rows, ring, Hkv, block_size, D] or null
    int window, ring;    // window tokens (0: none) and ring blocks (window / block_size + 1)
    int* status;
};

// One warp per (token, KV head, K|V) row; EPL = D / 32 values per lane.
template <typename T, int EPL, int QMODE>
__global__ void kv_append_quant_kernel(QuantArgs a) {
    const int lane = threadIdx.x & 31;
    const int64_t warps_total = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    const int64_t rows = static_cast<int64_t>(a.T) * a.hkv * 2;
    for (int64_t r = blockIdx.x * static_cast<int64_t>(blockDim.x >> 5) + (threadIdx.x >> 5);
         r < rows; r += warps_total) {
        const int which = static_cast<int>(r & 1);  // 0 = K, 1 = V
        const int64_t th = r >> 1;
        const int64_t t = th / a.hkv;
        const int h = static_cast<int>(th - t * a.hkv);
        const int64_t slot = a.slots[t];
        if (slot < 0) continue;
        if (slot >= a.num_slots) {
            if (lane == 0 && which == 0 && h == 0) atomicOr(a.status, PKV_STATUS_BAD_SLOT);
            continue;
        }
        const T* src = static_cast<const T*>(which ? a.v : a.k) +
                       (t * a.hkv + h) * static_cast<int64_t>(a.D) + lane * EPL;
        float x[EPL];
        load_row<T, EPL>(src, x);
        const int64_t blk = slot / a.block_size, off = slot - blk * a.block_size;
        const int64_t row = (blk * a.hkv + h) * a.block_size + off;  // (block, head, offset)

        if constexpr (QMODE == PKV_QMODE_INT4_ASYM) {
            const int lpg = a.group_size / EPL;  // lanes per group (power of two, <= 32)
            float mn = x[0], mx = x[0];
#pragma unroll
            for (int i = 1; i < EPL; ++i) {
                mn = fminf(mn, x[i]);
                mx = fmaxf(mx, x[i]);
            }
            for (int o = 1; o < lpg; o <<= 1) {
                mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            }
            __half s16 = f16_sat(__fdiv_rn(__fsub_rn(mx, mn), 15.0f));
            if (mx == mn || __half2float(s16) == 0.0f) s16 = __float2half_rn(1.0f);
            const float s = __half2float(s16);
            __half z16 = f16_sat(__fdiv_rn(-mn, s));
            if (__half2float(z16) == 0.0f) z16 = __float2half_rn(0.0f);  // -0 -> +0
            const float z = __half2float(z16);
            uint32_t packed = 0;
#pragma unroll
            for (int i = 0; i < EPL; ++i) {
                float qf = rintf(__fadd_rn(__fdiv_rn(x[i], s), z));
                qf = fminf(fmaxf(qf, 0.0f), 15.0f);
                packed |= static_cast<uint32_t>(qf) << (4 * i);
            }
            uint8_t* dst = a.codes[which] + row * (a.D / 2) + lane * (EPL / 2);
            if constexpr (EPL == 2) {
                *dst = static_cast<uint8_t>(packed);
            } else if constexpr (EPL == 4) {
                *reinterpret_cast<uint16_t*>(dst) = static_cast<uint16_t>(packed);
            } else {
                *reinterpret_cast<uint32_t*>(dst) = packed;
            }
            if ((lane & (lpg - 1)) == 0) {
                const int64_t gi = row * (a.D / a.group_size) + lane / lpg;
                a.scale[which][gi] = s16;
                a.zero[which][gi] = z16;
            }
        } else {  // FP8 E4M3, one scale per row
            float am = fabsf(x[0]);
#pragma unroll
            for (int i = 1; i < EPL; ++i) am = fmaxf(am, fabsf(x[i]));
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
            __half s16 = f16_sat(__fdiv_rn(am, 448.0f));
            if (__half2float(s16) == 0.0f) s16 = __float2half_rn(1.0f);
            const float s = __half2float(s16);
            uint32_t bytes[EPL / 2];
#pragma unroll
            for (int i = 0; i < EPL / 2; ++i) {
                const float y0 = __fdiv_rn(x[2 * i], s), y1 = __fdiv_rn(x[2 * i + 1], s);
                unsigned short pr;
                asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(pr) : "f"(y1), "f"(y0));
                bytes[i] = pr;
            }
            uint8_t* dst = a.codes[which] + row * a.D + lane * EPL;
            if constexpr (EPL == 2) {
                *reinterpret_cast<uint16_t*>(dst) = static_cast<uint16_t>(bytes[0]);
            } else if constexpr (EPL == 4) {
                *reinterpret_cast<uint32_t*>(dst) = bytes[0] | (bytes[1] << 16);
            } else {
                *reinterpret_cast<uint2*>(dst) =
                    make_uint2(bytes[0] | (bytes[1] << 16), bytes[2] | (bytes[3] << 16));
            }
            if (lane == 0) a.scale[which][row] = s16;
        }

        const int pos = a.positions[t];
        if (a.window > 0) {
            // every token passes through the 16-bit window ring of its
            // sequence; a token whose ring slot a later token of the same
            // call takes again (the entry one ring span ahead: same sequence,
            // position + span) is not written, so no two writes of one call
            // race on a slot
            const int sr = a.seq_idx[t];
            const int64_t span = static_cast<int64_t>(a.ring) * a.block_size;
            const bool superseded = t + span < a.T && a.seq_idx[t + span] == sr &&
                                    a.positions[t + span] == pos + span;
            if (pos < 0 || sr < 0 || sr >= a.sink_rows) {
                if (lane == 0) atomicOr(a.status, PKV_STATUS_BAD_SINK);
            } else if (!superseded) {
                const int64_t rb = (pos / a.block_size) % a.ring;
                T* dst = static_cast<T*>(a.win[which]) +
                         (((static_cast<int64_t>(sr) * a.ring + rb) * a.hkv + h) * a.block_size +
                          pos % a.block_size) * a.D +
                         lane * EPL;
                copy_row<T, EPL>(src, dst);
            }
        }
        if (pos < a.n_sink) {
            const int sr = a.seq_idx[t];
            if (pos < 0 || sr < 0 || sr >= a.sink_rows) {
                if (lane == 0) atomicOr(a.status, PKV_STATUS_BAD_SINK);
            } else {
                T* dst = static_cast<T*>(a.sink[which]) +
                         ((static_cast<int64_t>(sr) * a.n_sink + pos) * a.hkv + h) * a.D +
                         lane * EPL;
                copy_row<T, EPL>(src, dst);
            }
        }
    }
}

struct CopyArgs {
    uint4* pool[8];
    int64_t chunks[8];
};

__global__ void copy_blocks_kernel(CopyArgs a, const int32_t* __restrict__ pairs, int num_blocks,
                                   int* __restrict__ status) {
    const int pi = blockIdx.x, pl = blockIdx.y;
    const int src = pairs[2 * pi], dst = pairs[2 * pi + 1];
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
        if (threadIdx.x == 0 && pl == 0) atomicOr(status, PKV_STATUS_BAD_PAIR);
        return;
    }
    const int64_t n = a.chunks[pl];
    const uint4* s = a.pool[pl] + static_cast<int64_t>(src) * n;
    uint4* d = a.pool[pl] + static_cast<int64_t>(dst) * n;
    for (int64_t i = threadIdx.x; i < n; i += blockDim.x) d[i] = s[i];
}

int grid_for(int64_t work_items, int per_block) {
    int64_t g = (work_items + per_block - 1) / per_block;
    if (g < 1) g = 1;
    if (g > 152 * 16) g = 152 * 16;
    return static_cast<int>(g);
}

template <typename T, int EPL>
void launch_quant(const QuantArgs& a, int qmode, cudaStream_t s) {
    const int64_t rows = static_cast<int64_t>(a.T) * a.hkv * 2;
    const int grid = grid_for(rows, 8);
    if (qmode == PKV_QMODE_INT4_ASYM)
        kv_append_quant_kernel<T, EPL, PKV_QMODE_INT4_ASYM><<<grid, 256, 0, s>>>(a);
    else
        kv_append_quant_kernel<T, EPL, PKV_QMODE_FP8_E4M3><<<grid, 256, 0, s>>>(a);
}

}  // namespace
}  // namespace pkv

extern "C" int pkv_kv_append(const void* k, const void* v, const int64_t* slot_mapping,
                             int32_t num_tokens, void* k_pool, void* v_pool, int32_t num_blocks,
                             int32_t num_kv_heads, int32_t head_dim, int32_t block_size, int dtype,
                             void* stream) {
    if (num_tokens < 0 || num_blocks <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
        block_size <= 0 || head_dim % 8 != 0 || (dtype != PKV_DTYPE_F16 && dtype != PKV_DTYPE_BF16))
        return PKV_ERR_INVALID_ARG;
    if (num_tokens == 0) return PKV_OK;
    if (!k || !v || !slot_mapping || !k_pool || !v_pool) return PKV_ERR_INVALID_ARG;
    if (!pkv::aligned16(k) || !pkv::aligned16(v) || !pkv::aligned16(k_pool) ||
        !pkv::aligned16(v_pool) || (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
        return PKV_ERR_MISALIGNED;
    int* st = pkv::status_word();
    if (!st) return PKV_ERR_CUDA;
    const int cpr = head_dim / 8;  // 16-byte chunks per row
    const int64_t total = static_cast<int64_t>(num_tokens) * num_kv_heads * cpr;
    const int64_t num_slots = static_cast<int64_t>(num_blocks) * block_size;
    pkv::kv_append_kernel<<<pkv::grid_for(total, 256), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint4*>(k), static_cast<const uint4*>(v), slot_mapping, total,
        num_kv_heads, cpr, block_size, num_slots, static_cast<uint4*>(k_pool),
        static_cast<uint4*>(v_pool), st);
    return pkv::launch_status();
}

extern "C" int pkv_kv_append_quant(const void* k, const void* v, const int64_t* slot_mapping,
                                   const int32_t* positions, const int32_t* seq_idx,
                                   int32_t num_tokens, void* k_codes, void* k_scale, void* k_zero,
                                   void* v_codes, void* v_scale, void* v_zero, void* sink_k,
                                   void* sink_v, int32_t n_sink, int32_t sink_rows, void* win_k,
                                   void* win_v, int32_t window, int32_t num_blocks,
                                   int32_t num_kv_heads, int32_t head_dim,
                                   int32_t block_size, int32_t group_size, int qmode, int dtype,
                                   void* stream) {
    if (num_tokens < 0 || num_blocks <= 0 || num_kv_heads <= 0 || block_size <= 0 ||
        n_sink < 0 || window < 0 || (dtype != PKV_DTYPE_F16 && dtype != PKV_DTYPE_BF16))
        return PKV_ERR_INVALID_ARG;
    if (qmode != PKV_QMODE_INT4_ASYM && qmode != PKV_QMODE_FP8_E4M3) return PKV_ERR_INVALID_ARG;
    if (window % block_size != 0) return PKV_ERR_INVALID_ARG;
    if (head_dim != 64 && head_dim != 128 && head_dim != 256) return PKV_ERR_UNSUPPORTED;
    const int epl = head_dim / 32;
    if (qmode == PKV_QMODE_INT4_ASYM) {
        if (group_size <= 0 || head_dim % group_size != 0) return PKV_ERR_INVALID_ARG;
        const int lpg = group_size / epl;
        if (group_size % epl != 0 || lpg < 1 || lpg > 32 || (lpg & (lpg - 1)) != 0)
            return PKV_ERR_UNSUPPORTED;
    } else {
        group_size = head_dim;
    }
    if (num_tokens == 0) return PKV_OK;
    if (!k || !v || !slot_mapping || !positions || !seq_idx || !k_codes || !v_codes || !k_scale ||
        !v_scale)
        return PKV_ERR_INVALID_ARG;
    if (qmode == PKV_QMODE_INT4_ASYM && (!k_zero || !v_zero)) return PKV_ERR_INVALID_ARG;
    if (n_sink > 0 && (!sink_k || !sink_v || sink_rows <= 0)) return PKV_ERR_INVALID_ARG;
    if (window > 0 && (!win_k || !win_v || sink_rows <= 0)) return PKV_ERR_INVALID_ARG;
    if (window > 0 && (!pkv::aligned16(win_k) || !pkv::aligned16(win_v))) return PKV_ERR_MISALIGNED;
    if (!pkv::aligned16(k) || !pkv::aligned16(v) || !pkv::aligned16(k_codes) ||
        !pkv::aligned16(v_codes) || (n_sink > 0 && (!pkv::aligned16(sink_k) || !pkv::aligned16(sink_v))))
        return PKV_ERR_MISALIGNED;
    int* st = pkv::status_word();
    if (!st) return PKV_ERR_CUDA;
    pkv::QuantArgs a;
    a.k = k;
    a.v = v;
    a.slots = slot_mapping;
    a.positions = positions;
    a.seq_idx = seq_idx;
    a.T = num_tokens;
    a.hkv = num_kv_heads;
    a.D = head_dim;
    a.block_size = block_size;
    a.group_size = group_size;
    a.n_sink = n_sink;
    a.sink_rows = sink_rows;
    a.num_slots = static_cast<int64_t>(num_blocks) * block_size;
    a.codes[0] = static_cast<uint8_t*>(k_codes);
    a.codes[1] = static_cast<uint8_t*>(v_codes);
    a.scale[0] = static_cast<__half*>(k_scale);
    a.scale[1] = static_cast<__half*>(v_scale);
    a.zero[0] = static_cast<__half*>(k_zero);
    a.zero[1] = static_cast<__half*>(v_zero);
    a.sink[0] = sink_k;
    a.sink[1] = sink_v;
    a.win[0] = win_k;
    a.win[1] = win_v;
    a.window = window;
    a.ring = window / block_size + 1;
    a.status = st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (dtype == PKV_DTYPE_BF16) {
        if (epl == 2) pkv::launch_quant<__nv_bfloat16, 2>(a, qmode, s);
        else if (epl == 4) pkv::launch_quant<__nv_bfloat16, 4>(a, qmode, s);
        else pkv::launch_quant<__nv_bfloat16, 8>(a, qmode, s);
    } else {
        if (epl == 2) pkv::launch_quant<__half, 2>(a, qmode, s);
        else if (epl == 4) pkv::launch_quant<__half, 4>(a, qmode, s);
        else pkv::launch_quant<__half, 8>(a, qmode, s);
    }
    return pkv::launch_status();
}

extern "C" int pkv_copy_blocks(void* const* pools, const int64_t* bytes_per_block, int32_t n_pools,
                               const int32_t* pairs, int32_t n_pairs, int32_t num_blocks,
                               void* stream) {
    if (n_pairs < 0 || n_pools < 1 || n_pools > 8 || num_blocks <= 0 || !pools || !bytes_per_block)
        return PKV_ERR_INVALID_ARG;
    if (n_pairs == 0) return PKV_OK;
    if (!pairs) return PKV_ERR_INVALID_ARG;
    pkv::CopyArgs a;
    for (int i = 0; i < 8; ++i) {
        a.pool[i] = nullptr;
        a.chunks[i] = 0;
    }
    for (int i = 0; i < n_pools; ++i) {
        if (!pools[i] || bytes_per_block[i] <= 0 || bytes_per_block[i] % 16 != 0)
            return PKV_ERR_INVALID_ARG;
        if (!pkv::aligned16(pools[i])) return PKV_ERR_MISALIGNED;
        a.pool[i] = static_cast<uint4*>(pools[i]);
        a.chunks[i] = bytes_per_block[i] / 16;
    }
    int* st = pkv::status_word();
    if (!st) return PKV_ERR_CUDA;
    dim3 grid(n_pairs, n_pools);
    pkv::copy_blocks_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(a, pairs,
                                                                               num_blocks, st);
    return pkv::launch_status();
}
