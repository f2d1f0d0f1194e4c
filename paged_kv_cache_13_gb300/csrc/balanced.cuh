// Balanced split-K ("stream-K" over block-heads), shared by the 16-bit and
// the quantised decode kernels.
//
// The work of one decode call is the ordered list of (sequence, KV head,
// 16-token unit) items -- sequence-major, then KV head, then unit --
// W = Hkv * sum_b ceil(ctx_b / 16) items (a unit is one block at the
// default block size of 16, half a 32-token block, or two 8-token blocks).
// Warp i of nwt = min(launched warps, W / min_items) takes the contiguous
// range [i W / nwt, (i + 1) W / nwt), so every warp streams the same number
// of units whatever the mix of context lengths: no wave quantisation, no
// short last partitions, one prologue per warp.  A range falls into runs of one (sequence, KV head); a warp writes
// one fp32 partial (m, l, o) per run it touches, at slot i + b * Hkv + kvh
// (rows slot * G + h of the partial arrays): the warps touching one run are
// consecutive and every range is non-empty, so slots never collide, and
// fewer than nwt + batch * Hkv slots are used.
#pragma once

#include "common.cuh"

namespace pkv {

constexpr int kSplitBS = 16;  // tokens per item (the kernels' token tile)

// Batches up to this size may use the balanced split (every warp scans the
// context lengths once).
constexpr int kBalancedMaxBatch = 1024;
// Fewest (sequence, KV head, unit) items a warp of the balanced split takes.
constexpr int kBalancedMinItems = 2;
// The automatic split is balanced when the tables could hold this many items
// per launched warp: below it fixed partitions measured as fast or faster
// (the balanced split's per-warp scan, partial rows and merge cost more than
// the wave quantisation they remove).
constexpr int kBalancedItemsPerWarp = 32;

// SM count of the current device (152 when it cannot be queried), cached.
int num_sms();
// Warps a balanced split launches: warps_per_sm per SM (all resident at
// once), fewer for small problems.
int balanced_warps(int64_t max_items, int warps_per_sm);
// The most warps per SM any balanced kernel launches (the workspace bound).
constexpr int kBalancedMaxWarpsPerSm = 20;
// Whether an automatic split may be balanced for at most max_items items.
bool balanced_candidate(int64_t batch, int64_t max_items);
// Whether an automatic split over tables of max_units 16-token units is
// balanced.
bool use_balanced(int64_t batch, int64_t hkv, int64_t max_units);
// Workspace bytes of a balanced split: nwt * G + batch * hq partial rows.
size_t balanced_bytes(int32_t batch, int32_t hq, int32_t G, int32_t D, int32_t nwt);
// The merge of a balanced split (decode.cu), launched behind the split
// kernel with programmatic dependent launch; out has the 16-bit dtype.  cap:
// the tables' capacity in tokens (max_blocks * block_size).
int launch_balanced_merge(const int32_t* ctx_lens, int batch, int hq, int hkv, int D, int cap,
                          int nwt, const float* ws_o, const float* ws_ml, void* out, int dtype,
                          cudaStream_t st);

__device__ __forceinline__ int blocks_of(int ctx, int cap) {
    ctx = ctx < 0 ? 0 : (ctx > cap ? cap : ctx);
    return (ctx + kSplitBS - 1) / kSplitBS;
}

// Log-sum-exp merge of the partition partials q = q0, q0 + step, ... < np of
// one (sequence, query head, column): each partial holds (m_q, l_q, o_q[d])
// with o_q unnormalised.  Loads of 8 partitions are issued together, then
// folded into a running (M, L, acc) with one rescale per chunk.  Partials
// are read from L2 (.cg): they were written by another grid.
struct MergeAcc {
    float M, L, acc;
};

__device__ __forceinline__ MergeAcc merge_range(const float* __restrict__ ml, int64_t stride_ml,
                                                const float* __restrict__ ov, int64_t stride_o,
                                                int q0, int np, int step) {
    MergeAcc r{neg_inf(), 0.f, 0.f};
    for (int qa = q0; qa < np; qa += 8 * step) {
        float mq[8], lq[8], oq[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int q = qa + j * step;
            const bool v = q < np;
            mq[j] = v ? __ldcg(ml + q * stride_ml) : neg_inf();
            lq[j] = v ? __ldcg(ml + q * stride_ml + 1) : 0.f;
            oq[j] = v ? __ldcg(ov + q * stride_o) : 0.f;
        }
        float mx = r.M;
#pragma unroll
        for (int j = 0; j < 8; ++j) mx = fmaxf(mx, mq[j]);
        if (mx == neg_inf()) continue;  // every partition so far was empty
        const float sc = ex2(r.M - mx);  // 0 while M is still -inf
        r.acc *= sc;
        r.L *= sc;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float w = ex2(mq[j] - mx);
            r.acc += w * oq[j];
            r.L += w * lq[j];
        }
        r.M = mx;
    }
    return r;
}

// First warp of a balanced split whose range holds item x: the largest i
// with floor(i W / nwt) <= x.
__device__ __forceinline__ int64_t first_warp(int64_t x, int64_t W, int64_t nwt) {
    return ((x + 1) * nwt - 1) / W;
}

// One warp's range, walked run by run.  The host keeps
// batch * Hkv * (units per table) below 2^30, so item indices fit in int.
struct WarpSplit {
    const int32_t* ctx_lens;
    int cap, hkv;
    int pos, E;    // remaining items [pos, E)
    int b, nb, cs; // current sequence, its unit count, its first item
    // current run segment: sequence b, KV head kvh, units [lb0, lb1)
    int ctx, kvh, lb0, lb1;

    // Sets up warp i's range; false when it has none.  Every lane of the warp
    // calls it (warp-collective).  cap_tokens: the tables' capacity
    // (max_blocks * block_size); bad: some context length was outside
    // [0, cap_tokens].
    __device__ __forceinline__ bool begin(const int32_t* lens, int batch, int cap_tokens, int hkv_,
                                          int nwt_launch, int min_items, int i, bool& bad) {
        const int lane = threadIdx.x & 31;
        ctx_lens = lens;
        cap = cap_tokens;
        hkv = hkv_;
        int mine = 0;
        bad = false;
        for (int j = lane; j < batch; j += 32) {
            const int x = lens[j];
            bad |= x < 0 || x > cap;
            mine += blocks_of(x, cap);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) mine += __shfl_xor_sync(0xffffffffu, mine, off);
        bad = __any_sync(0xffffffffu, bad);
        const int W = mine * hkv;
        const int nwt = max(min(W / min_items, nwt_launch), 1);
        if (W == 0 || i >= nwt) return false;
        pos = static_cast<int>(static_cast<int64_t>(i) * W / nwt);
        E = static_cast<int>(static_cast<int64_t>(i + 1) * W / nwt);
        // the sequence holding item pos
        b = nb = cs = 0;
        int run = 0;
        for (int base = 0; base < batch; base += 32) {
            const int j = base + lane;
            const int nbj = j < batch ? blocks_of(lens[j], cap) : 0;
            int incl = nbj;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += y;
            }
            const unsigned hit = __ballot_sync(0xffffffffu, j < batch && pos < (run + incl) * hkv);
            if (hit) {
                const int src = __ffs(hit) - 1;
                b = base + src;
                nb = __shfl_sync(0xffffffffu, nbj, src);
                cs = (run + __shfl_sync(0xffffffffu, incl - nbj, src)) * hkv;
                break;
            }
            run += __shfl_sync(0xffffffffu, incl, 31);
        }
        return true;
    }

    // Advances to the next run segment of the range; false at its end.
    __device__ __forceinline__ bool next() {
        if (pos >= E) return false;
        while (pos >= cs + nb * hkv) {  // next non-empty sequence
            cs += nb * hkv;
            ++b;
            nb = blocks_of(ctx_lens[b], cap);
        }
        ctx = min(max(ctx_lens[b], 0), cap);
        kvh = (pos - cs) / nb;
        lb0 = pos - cs - kvh * nb;
        lb1 = min(nb, lb0 + (E - pos));
        pos += lb1 - lb0;
        return true;
    }
};

}  // namespace pkv
