// Paged single-query GQA decode attention over a 16-bit (bf16 / fp16) cache.
//
// What it computes: for sequence b and query head h (KV head h / G),
//   out[b, h] = sum_t softmax_t(scale * <q[b, h], K_t>) V_t,  t < ctx_b,
// with K_t, V_t gathered through the block table ("The 8GB VRAM
// Breakthrough", §3 "How Logical-to-Physical Block Tables Work": the kernel
// reads the table on the fly and gathers the non-contiguous physical blocks
// for QK^T and the softmax-weighted sum of V).  Optionally the same kernel
// first writes the decode step's new K/V row into its slot (the KV-append of
// §1, "write one new KV vector back"), taking that row from the inputs
// instead of reading it back.
//
// Design (sm_103a):
// * Work unit = (sequence, KV head, partition of `part_blocks` blocks).  One
//   CTA of NW warps per unit; the warps take the partition's blocks
//   round-robin, each keeping its own online-softmax state (running max m,
//   sum l, accumulator o) for the G query heads of the KV head; the CTA merges
//   its warps through shared memory at the end.  With several partitions per
//   sequence (flash-decoding split-K) each CTA writes an fp32 (m, l, o)
//   partial and a merge kernel, launched behind it with programmatic
//   dependent launch, combines the partials with a log-sum-exp rescale.
// * Each warp loads the physical ids of all its blocks with one coalesced
//   load (lane k holds the id of the warp's k-th block), so a block's K/V
//   loads never wait behind a table load.
// * The token tile is a 16-token unit.  At the default block size of 16 a
//   unit is one block; at 32 it is half a block; at 8 it is two blocks, so
//   its rows 0-7 and 8-15 come from two table entries.  Either way a unit's
//   rows of one KV head are two runs of 8 x D contiguous 16-bit values (one
//   16 x D run, 4 KiB for D = 128, at block sizes 16 and 32).  Each lane issues 16-byte loads straight from global memory
//   into registers, shaped so that the registers ARE the tensor-core fragments
//   (no shared-memory staging, no shuffles of K or V):
//     QK^T : S^T[16 tok x 8 heads] = K[16 x D] . Q^T[D x 8]   (mma m16n8k16,
//            tokens as M, the GQA group as N, head dim as K).  Lane (g, c)
//            (g = lane / 4, c = lane % 4) loads K rows g and g+8 at
//            [32i + 8c, +8): a 16-byte piece whose four 32-bit words are the
//            A-fragment registers of two k-steps.  The k order inside a
//            k-step is permuted, and Q's B fragment uses the same permutation.
//     PV   : O^T[D x 8 heads] = V^T[D x 16 tok] . P^T[16 tok x 8]  (head dim
//            as M, heads as N, tokens as K).  Lane (g, c) loads V rows
//            2c, 2c+1, 8+2c, 9+2c at [64j + 8g, +8); one byte-permute per
//            register pairs two tokens of the same column into the A fragment.
//            P^T comes from the QK^T accumulator by one 8x8 movmatrix
//            transpose per half-block.
//   Heads beyond G in the N dimension carry zero queries and are ignored.
// * Online softmax in base 2 (logits pre-multiplied by scale * log2 e);
//   block max by three xor-shuffles across the 8 token lanes; the running sum
//   stays a per-lane partial until the end.
// * Tokens at or past ctx in the last block get logit -inf, and their V rows
//   are zeroed in registers (an unwritten slot may hold NaN bit patterns).

#include <atomic>
#include <type_traits>

#include "balanced.cuh"

namespace pkv {
namespace {

constexpr int kUnit = 16;  // tokens per unit: the kernels' token tile (block sizes 8, 16, 32)
constexpr int kNW = 4;  // warps per CTA (4 beat 8 in a sweep on the 64-sequence layer)
constexpr float kLog2e = 1.4426950408889634f;
// Headroom (log2 units) a logit may rise above the running reference max
// before the online softmax rescales: weights stay <= 2^8.
constexpr float kSlack = 8.f;

enum Mode { kSingle = 0, kPartials = 1 };

struct DecodeArgs {
    const void* q;
    const void* k_pool;
    const void* v_pool;
    void* k_pool_w;        // writable views of the pools (fused append)
    void* v_pool_w;
    const void* k_new;     // [B, Hkv, D] new rows (fused append)
    const void* v_new;
    const int64_t* slots;  // [B] slot of each new row (fused append)
    const int32_t* tables;
    const int32_t* ctx_lens;
    int hq, hkv, G, num_blocks, max_blocks, part_blocks, max_parts;
    int cap;  // table capacity in tokens: max_blocks * block_size
    float scale_log2;
    void* out;
    float* ws_o;   // [B, Hq, max_parts, D]
    float* ws_ml;  // [B, Hq, max_parts, 2]
    int* status;
};

// Element e (0 .. D/8-1) of lane group g in the PV fragment layout sits at
// head-dim column 64 * (e / 8) + 8 * g + e % 8.
__device__ __forceinline__ int pv_col(int e, int g) { return 64 * (e >> 3) + 8 * g + (e & 7); }

// Whether P enters the PV product as two 16-bit terms (value + residual).
template <typename T>
constexpr bool kSplitP = false;
template <>
constexpr bool kSplitP<__nv_bfloat16> = true;

// The bf16 halves of a packed pair, as floats (exact).
__device__ __forceinline__ float lo_float(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float hi_float(uint32_t x) { return __uint_as_float(x & 0xffff0000u); }

// Online-softmax state of one warp for the query heads 2c, 2c+1 of its lanes.
template <int MT>
struct WarpState {
    float m0, m1, l0, l1;
    float o[MT][4];
};

// 16-byte shared-memory load at a shared-window address, kept in place (not
// hoisted out of the block loop, so the query fragments cost no registers).
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 r;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "r"(addr));
    return r;
}

// Query fragment sources for attend_block: registers, or this warp's
// shared slice re-read for every block (16 fewer live registers).
template <int KC>
struct QRegs {
    uint4 f[KC];
    __device__ __forceinline__ uint4 get(int i) const { return f[i]; }
};
struct QShared {
    uint32_t addr;
    __device__ __forceinline__ uint4 get(int i) const { return lds128(addr + i * 512); }
};

// Q^T B-fragments of KV head kvh's query group, staged in this warp's
// shared slice: lane (g, c) holds query head g's columns [32i + 8c, +8) at
// slot[i * 32] (zero for g >= G).  Returns the lane's shared address.
template <typename T, int D>
__device__ __forceinline__ uint32_t stage_query(const DecodeArgs& a, int b, int kvh, int g, int c,
                                                uint4* slot) {
    constexpr int KC = D / 32;
    if (g < a.G) {
        const T* qrow = static_cast<const T*>(a.q) + (static_cast<int64_t>(b) * a.hq + kvh * a.G + g) * D;
#pragma unroll
        for (int i = 0; i < KC; ++i) slot[i * 32] = *reinterpret_cast<const uint4*>(qrow + 32 * i + 8 * c);
    } else {
#pragma unroll
        for (int i = 0; i < KC; ++i) slot[i * 32] = make_uint4(0, 0, 0, 0);
    }
    __syncwarp();
    return static_cast<uint32_t>(__cvta_generic_to_shared(slot));
}

// Table entries of 16-token unit u of a sequence at block size BS: entry u
// (BS 16); entry u / 2, from its row 16 (u % 2) (BS 32); entries 2u and
// 2u + 1 (BS 8), the second only while it holds context tokens (nent:
// entries the context covers) -- past it the first stands in, its rows
// being masked.
template <int BS>
struct UnitIds {
    int e0, e1;
    __device__ __forceinline__ void load(const int32_t* trow, int u, bool in, int nent) {
        e0 = e1 = 0;
        if (!in) return;
        if constexpr (BS == 8) {
            e0 = trow[2 * u];
            e1 = 2 * u + 1 < nent ? trow[2 * u + 1] : e0;
        } else {
            e0 = trow[u * kUnit / BS];
        }
    }
    // lane src's entries
    __device__ __forceinline__ UnitIds shfl(int src) const {
        UnitIds r;
        r.e0 = __shfl_sync(0xffffffffu, e0, src);
        r.e1 = BS == 8 ? __shfl_sync(0xffffffffu, e1, src) : 0;
        return r;
    }
    __device__ __forceinline__ bool valid(int num_blocks) const {
        return static_cast<unsigned>(e0) < static_cast<unsigned>(num_blocks) &&
               (BS != 8 || static_cast<unsigned>(e1) < static_cast<unsigned>(num_blocks));
    }
    // Element offsets, within a pool, of the unit's rows 0-7 (lo) and 8-15
    // (hi) of KV head kvh.
    template <int D>
    __device__ __forceinline__ void bases(int hkv, int kvh, int u, int64_t& lo, int64_t& hi) const {
        lo = (static_cast<int64_t>(e0) * hkv + kvh) * (BS * D);
        if constexpr (BS == 32) lo += (u & 1) * (kUnit * D);
        if constexpr (BS == 8) {
            hi = (static_cast<int64_t>(e1) * hkv + kvh) * (BS * D);
        } else {
            hi = lo + 8 * D;
        }
    }
};

// Attend one 16-token unit (logical index lb; rows 0-7 at pool offset lo,
// rows 8-15 at hi) into the warp state.  INJECT: row app_off of the unit is
// the decode step's new row; it is taken from the inputs (and stored to the
// pool) instead of the loads.
template <typename T, int D, bool INJECT, typename QS>
__device__ __forceinline__ void attend_block(const DecodeArgs& a, int b, int kvh, int lb, int64_t lo,
                                             int64_t hi, int ctx, int app_off, const QS& qs,
                                             WarpState<D / 16>& w, int g, int c) {
    using H = Half16<T>;
    constexpr int KC = D / 32;
    constexpr int VC = D / 64;
    constexpr int MT = D / 16;
    const int vrow0 = 2 * c, vrow1 = 2 * c + 1, vrow2 = 8 + 2 * c, vrow3 = 9 + 2 * c;
    const T* kp = static_cast<const T*>(a.k_pool);
    const T* vpl = static_cast<const T*>(a.v_pool);
    // Row sources: the pool, except that with INJECT the lanes holding row
    // app_off read the decode step's new row from the inputs instead.
    const T* kr0p = kp + lo + g * D;
    const T* kr1p = kp + hi + g * D;
    const T* vp0 = vpl + lo + vrow0 * D;
    const T* vp1 = vpl + lo + vrow1 * D;
    const T* vp2 = vpl + hi + (vrow2 - 8) * D;
    const T* vp3 = vpl + hi + (vrow3 - 8) * D;
    if constexpr (INJECT) {
        const int64_t nrow = (static_cast<int64_t>(b) * a.hkv + kvh) * D;
        const T* kn = static_cast<const T*>(a.k_new) + nrow;
        const T* vn = static_cast<const T*>(a.v_new) + nrow;
        if (g == app_off) kr0p = kn;
        if (g + 8 == app_off) kr1p = kn;
        if (vrow0 == app_off) vp0 = vn;
        if (vrow1 == app_off) vp1 = vn;
        if (vrow2 == app_off) vp2 = vn;
        if (vrow3 == app_off) vp3 = vn;
    }

    uint4 kr0[KC], kr1[KC], vr[4][VC];
#pragma unroll
    for (int i = 0; i < KC; ++i) {
        kr0[i] = ldg_stream(kr0p + 32 * i + 8 * c);
        kr1[i] = ldg_stream(kr1p + 32 * i + 8 * c);
    }
#pragma unroll
    for (int j = 0; j < VC; ++j) {
        vr[0][j] = ldg_stream(vp0 + 64 * j + 8 * g);
        vr[1][j] = ldg_stream(vp1 + 64 * j + 8 * g);
        vr[2][j] = ldg_stream(vp2 + 64 * j + 8 * g);
        vr[3][j] = ldg_stream(vp3 + 64 * j + 8 * g);
    }

    if constexpr (INJECT) {
        // Store the new row to the pool from the lanes that hold its pieces
        // (each 16-byte piece exactly once).
        const int64_t row = app_off < 8 ? lo + app_off * D : hi + (app_off - 8) * D;
        T* kw = static_cast<T*>(a.k_pool_w) + row;
        T* vw = static_cast<T*>(a.v_pool_w) + row;
#pragma unroll
        for (int i = 0; i < KC; ++i) {
            if (g == app_off) *reinterpret_cast<uint4*>(kw + 32 * i + 8 * c) = kr0[i];
            if (g + 8 == app_off) *reinterpret_cast<uint4*>(kw + 32 * i + 8 * c) = kr1[i];
        }
#pragma unroll
        for (int j = 0; j < VC; ++j) {
            if (vrow0 == app_off) *reinterpret_cast<uint4*>(vw + 64 * j + 8 * g) = vr[0][j];
            if (vrow1 == app_off) *reinterpret_cast<uint4*>(vw + 64 * j + 8 * g) = vr[1][j];
            if (vrow2 == app_off) *reinterpret_cast<uint4*>(vw + 64 * j + 8 * g) = vr[2][j];
            if (vrow3 == app_off) *reinterpret_cast<uint4*>(vw + 64 * j + 8 * g) = vr[3][j];
        }
    }

    // ---- S^T = K Q^T: s[0]=S(t=g,h=2c) s[1]=S(g,2c+1) s[2]=S(g+8,2c) s[3]=S(g+8,2c+1)
    float s[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < KC; ++i) {
        const uint4 qf = qs.get(i);
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            H::mma(s, word(kr0[i], 2 * e), word(kr1[i], 2 * e), word(kr0[i], 2 * e + 1),
                   word(kr1[i], 2 * e + 1), word(qf, 2 * e), word(qf, 2 * e + 1));
        }
    }
    const int tok0 = lb * kUnit + g;
    const bool ok0 = tok0 < ctx, ok1 = tok0 + 8 < ctx;
    const float x0 = ok0 ? s[0] * a.scale_log2 : neg_inf();
    const float x1 = ok0 ? s[1] * a.scale_log2 : neg_inf();
    const float x2 = ok1 ? s[2] * a.scale_log2 : neg_inf();
    const float x3 = ok1 ? s[3] * a.scale_log2 : neg_inf();

    // ---- online softmax (base 2); heads 2c (x0, x2) and 2c+1 (x1, x3).
    // The reference max m is raised only when a logit of this block exceeds
    // it by more than kSlack; otherwise the weights 2^(x - m) <= 2^kSlack are
    // taken against the old m, skipping the warp-wide max and the rescale of
    // o and l (any reference works: m cancels in o / l and in the merges).
    const float bx0 = fmaxf(x0, x2), bx1 = fmaxf(x1, x3);
    if (__any_sync(0xffffffffu, bx0 > w.m0 + kSlack || bx1 > w.m1 + kSlack)) {
        float bm0 = bx0, bm1 = bx1;
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            bm0 = fmaxf(bm0, __shfl_xor_sync(0xffffffffu, bm0, off));
            bm1 = fmaxf(bm1, __shfl_xor_sync(0xffffffffu, bm1, off));
        }
        const float mn0 = fmaxf(w.m0, bm0), mn1 = fmaxf(w.m1, bm1);
        const float al0 = ex2(w.m0 - mn0), al1 = ex2(w.m1 - mn1);
        w.l0 *= al0;
        w.l1 *= al1;
        w.m0 = mn0;
        w.m1 = mn1;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            w.o[mt][0] *= al0;
            w.o[mt][1] *= al1;
            w.o[mt][2] *= al0;
            w.o[mt][3] *= al1;
        }
    }
    const float p0 = ex2(x0 - w.m0), p1 = ex2(x1 - w.m1);
    const float p2 = ex2(x2 - w.m0), p3 = ex2(x3 - w.m1);
    w.l0 += p0 + p2;
    w.l1 += p1 + p3;
    // P^T B-fragments: transpose the two 8x8 (token x head) halves.  bf16
    // keeps 8 bits of P, which alone can move a short context's output by
    // ~2e-3; there P also goes in as a second bf16 term, its rounding
    // residual, so the products see ~16 bits of P (fp16's 11 suffice).
    const uint32_t h01 = H::pack(p0, p1), h23 = H::pack(p2, p3);
    const uint32_t pb0 = movmatrix_trans(h01);
    const uint32_t pb1 = movmatrix_trans(h23);
    uint32_t pr0 = 0, pr1 = 0;
    if constexpr (kSplitP<T>) {
        pr0 = movmatrix_trans(H::pack(p0 - lo_float(h01), p1 - hi_float(h01)));
        pr1 = movmatrix_trans(H::pack(p2 - lo_float(h23), p3 - hi_float(h23)));
    }

    if (lb * kUnit + kUnit > ctx) {  // last, partial unit: zero masked V rows
        const int t0 = lb * kUnit;
#pragma unroll
        for (int j = 0; j < VC; ++j) {
            if (t0 + vrow0 >= ctx) vr[0][j] = make_uint4(0, 0, 0, 0);
            if (t0 + vrow1 >= ctx) vr[1][j] = make_uint4(0, 0, 0, 0);
            if (t0 + vrow2 >= ctx) vr[2][j] = make_uint4(0, 0, 0, 0);
            if (t0 + vrow3 >= ctx) vr[3][j] = make_uint4(0, 0, 0, 0);
        }
    }

    // ---- O^T += V^T P^T
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
        constexpr int HALF = D / 16;
        const int elo = mt, ehi = mt + HALF;
        const int jl = elo >> 3, wl = (elo & 7) >> 1, hl = elo & 1;
        const int jh = ehi >> 3, wh = (ehi & 7) >> 1, hh = ehi & 1;
        const uint32_t sl = hl ? 0x7632u : 0x5410u;
        const uint32_t sh = hh ? 0x7632u : 0x5410u;
        const uint32_t a0 = __byte_perm(word(vr[0][jl], wl), word(vr[1][jl], wl), sl);
        const uint32_t a1 = __byte_perm(word(vr[0][jh], wh), word(vr[1][jh], wh), sh);
        const uint32_t a2 = __byte_perm(word(vr[2][jl], wl), word(vr[3][jl], wl), sl);
        const uint32_t a3 = __byte_perm(word(vr[2][jh], wh), word(vr[3][jh], wh), sh);
        H::mma(w.o[mt], a0, a1, a2, a3, pb0, pb1);
        if constexpr (kSplitP<T>) H::mma(w.o[mt], a0, a1, a2, a3, pr0, pr1);
    }
}

// The fused append's unit: its table entry holding the new row was checked
// against the slot, but at block size 8 the unit's other entry was not, so
// the entries are checked again here (a bad one skips the unit, store
// included, and flags the status).
template <typename T, int D, int BS, typename QS>
__device__ __forceinline__ void attend_appended(const DecodeArgs& a, int b, int kvh, int lb,
                                                const int32_t* trow, int nent, int ctx, int app_off,
                                                const QS& qs, WarpState<D / 16>& w, int g, int c) {
    UnitIds<BS> e;
    e.load(trow, lb, true, nent);
    if (!e.valid(a.num_blocks)) {
        if ((threadIdx.x & 31) == 0) atomicOr(a.status, PKV_STATUS_BAD_BLOCK);
        return;
    }
    int64_t lo, hi;
    e.template bases<D>(a.hkv, kvh, lb, lo, hi);
    attend_block<T, D, true>(a, b, kvh, lb, lo, hi, ctx, app_off, qs, w, g, c);
}

// Merge the NW warps' online-softmax states of one CTA through shared memory
// and pass each query head h < G, column d result -- unnormalised output
// acc, max M, sum L -- to store(h, d, acc, M, L).  Ends with a barrier, so
// the shared arrays may be reused right after.
template <int D, int NW, typename Store>
__device__ __forceinline__ void cta_merge(const WarpState<D / 16>& ws, int warp, int g, int c, int G,
                                          float (&sm_ml)[NW][8][2], float (&sm_o)[NW][8][D],
                                          Store store) {
    constexpr int MT = D / 16;
    float l0 = ws.l0, l1 = ws.l1;
    // finish the per-lane partial sums over the 8 token lanes
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, off);
        l1 += __shfl_xor_sync(0xffffffffu, l1, off);
    }
    if (g == 0) {
        sm_ml[warp][2 * c][0] = ws.m0;
        sm_ml[warp][2 * c][1] = l0;
        sm_ml[warp][2 * c + 1][0] = ws.m1;
        sm_ml[warp][2 * c + 1][1] = l1;
    }
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
        const int dl = pv_col(mt, g), dh = pv_col(mt + D / 16, g);
        sm_o[warp][2 * c][dl] = ws.o[mt][0];
        sm_o[warp][2 * c + 1][dl] = ws.o[mt][1];
        sm_o[warp][2 * c][dh] = ws.o[mt][2];
        sm_o[warp][2 * c + 1][dh] = ws.o[mt][3];
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < G * D; idx += NW * 32) {
        const int h = idx / D, d = idx - h * D;
        float M = neg_inf();
#pragma unroll
        for (int w = 0; w < NW; ++w) M = fmaxf(M, sm_ml[w][h][0]);
        float acc = 0.f, L = 0.f;
        if (M != neg_inf()) {
#pragma unroll
            for (int w = 0; w < NW; ++w) {
                const float sc = ex2(sm_ml[w][h][0] - M);
                acc += sc * sm_o[w][h][d];
                L += sc * sm_ml[w][h][1];
            }
        }
        store(h, d, acc, M, L);
    }
    __syncthreads();
}

template <typename T, int D, int NW, int MODE, bool APPEND, int BS>
__global__ void __launch_bounds__(NW * 32, 16 / NW) paged_decode_kernel(DecodeArgs a) {
    using H = Half16<T>;
    constexpr int KC = D / 32;  // 16-byte K pieces per lane per row
    constexpr int MT = D / 16;  // PV m-tiles

    const int p = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, c = lane & 3;

    int ctx = a.ctx_lens[b];
    const int cap = a.cap;
    if (ctx < 0 || ctx > cap) {
        if (threadIdx.x == 0 && p == 0 && kvh == 0) atomicOr(a.status, PKV_STATUS_BAD_CONTEXT);
        ctx = ctx < 0 ? 0 : cap;
    }
    const int nblk = (ctx + kUnit - 1) / kUnit;  // units
    const int nent = (ctx + BS - 1) / BS;        // table entries
    const int nparts = MODE == kSingle ? 1 : max((nblk + a.part_blocks - 1) / a.part_blocks, 1);
    if constexpr (MODE == kPartials) {
        // let the merge grid (launched with programmatic serialization) be
        // scheduled while this grid drains; it waits for our completion
        asm volatile("griddepcontrol.launch_dependents;");
    }
    if (p >= nparts) return;
    const int blk_begin = MODE == kSingle ? 0 : p * a.part_blocks;
    const int blk_end = MODE == kSingle ? nblk : min(blk_begin + a.part_blocks, nblk);
    const int32_t* trow = a.tables + static_cast<int64_t>(b) * a.max_blocks;

    // fused append: the new row belongs at logical position ctx - 1
    int app_lb = -1, app_off = 0;
    if constexpr (APPEND) {
        const int64_t slot = ctx > 0 ? a.slots[b] : -1;
        if (slot >= 0) {
            const int lb_last = (ctx - 1) / kUnit;
            if (lb_last >= blk_begin && lb_last < blk_end) {
                const int phys = trow[(ctx - 1) / BS], off = (ctx - 1) % BS;
                if (static_cast<unsigned>(phys) < static_cast<unsigned>(a.num_blocks) &&
                    slot == static_cast<int64_t>(phys) * BS + off) {
                    app_lb = lb_last;
                    app_off = (ctx - 1) % kUnit;
                } else if (threadIdx.x == 0) {
                    atomicOr(a.status, PKV_STATUS_BAD_SLOT);
                }
            }
        }
    }

    // Q^T B-fragments: lane (g, c) holds query head g's columns [32i + 8c, +8).
    __shared__ uint4 sm_q[NW][KC][32];
    const QShared qs{stage_query<T, D>(a, b, kvh, g, c, &sm_q[warp][0][lane])};

    WarpState<MT> ws;
    ws.m0 = ws.m1 = neg_inf();
    ws.l0 = ws.l1 = 0.f;
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) ws.o[mt][0] = ws.o[mt][1] = ws.o[mt][2] = ws.o[mt][3] = 0.f;

    // The appended unit, if any, is the last unit of this partition and so
    // the last one its warp visits: the loop stops there and the unit is
    // attended after the loop with the injection.
    UnitIds<BS> tab;
    tab.e0 = tab.e1 = 0;
    int k = 0, lb = blk_begin + warp;
    for (; lb < blk_end && lb != app_lb; ++k, lb += NW) {
        if ((k & 31) == 0) {  // table entries of this warp's next 32 units
            const int idx = lb + NW * lane;
            tab.load(trow, idx, idx < blk_end, nent);
        }
        const UnitIds<BS> e = tab.shfl(k & 31);
        if (!e.valid(a.num_blocks)) {
            if (lane == 0) atomicOr(a.status, PKV_STATUS_BAD_BLOCK);
            continue;
        }
        int64_t lo, hi;
        e.template bases<D>(a.hkv, kvh, lb, lo, hi);
        attend_block<T, D, false>(a, b, kvh, lb, lo, hi, ctx, 0, qs, ws, g, c);
    }
    if constexpr (APPEND) {
        if (lb == app_lb) attend_appended<T, D, BS>(a, b, kvh, lb, trow, nent, ctx, app_off, qs, ws, g, c);
    }
    __shared__ float sm_ml[NW][8][2];
    __shared__ float sm_o[NW][8][D];
    cta_merge<D, NW>(ws, warp, g, c, a.G, sm_ml, sm_o, [&](int h, int d, float acc, float M, float L) {
        const int64_t qh = static_cast<int64_t>(b) * a.hq + kvh * a.G + h;
        if constexpr (MODE == kSingle) {
            static_cast<T*>(a.out)[qh * D + d] = H::from_float(L > 0.f ? acc / L : 0.f);
        } else {
            const int64_t row = qh * a.max_parts + p;
            a.ws_o[row * D + d] = acc;
            if (d == 0) {
                a.ws_ml[2 * row] = M;
                a.ws_ml[2 * row + 1] = L;
            }
        }
    });
}

// Balanced split-K kernel for the 16-bit cache (the split itself:
// balanced.cuh).  Warp i walks its range run by run; within a run it
// attends its blocks in order, then writes the run's partial.  No barrier.
template <typename T, int D, bool APPEND, int BS>
__global__ void __launch_bounds__(kNW * 32, 16 / kNW)
    paged_decode_balanced_kernel(DecodeArgs a, int batch, int nwt_launch, int min_items) {
    constexpr int KC = D / 32;
    constexpr int MT = D / 16;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, c = lane & 3;
    // the merge grid may be scheduled now; it waits for this grid to finish
    asm volatile("griddepcontrol.launch_dependents;");
    __shared__ __align__(16) float sm_o[kNW][8][D];
    __shared__ uint4 sm_q[kNW][KC][32];

    const int i = blockIdx.x * kNW + warp;
    WarpSplit ws_;
    bool bad = false;
    const bool any = ws_.begin(a.ctx_lens, batch, a.cap, a.hkv, nwt_launch, min_items, i, bad);
    if (i == 0 && bad && lane == 0) atomicOr(a.status, PKV_STATUS_BAD_CONTEXT);
    if (!any) return;

    while (ws_.next()) {
        const int b = ws_.b, nb = ws_.nb, ctx = ws_.ctx, kvh = ws_.kvh, lb0 = ws_.lb0, lb1 = ws_.lb1;
        const int32_t* trow = a.tables + static_cast<int64_t>(b) * a.max_blocks;
        const int nent = (ctx + BS - 1) / BS;  // table entries the context covers

        // fused append: the new row is at ctx - 1, in the run's last unit
        int app_lb = -1, app_off = 0;
        if constexpr (APPEND) {
            if (lb1 == nb) {
                const int64_t slot = a.slots[b];
                if (slot >= 0) {
                    const int phys = trow[nent - 1], off = (ctx - 1) % BS;
                    if (static_cast<unsigned>(phys) < static_cast<unsigned>(a.num_blocks) &&
                        slot == static_cast<int64_t>(phys) * BS + off) {
                        app_lb = nb - 1;
                        app_off = (ctx - 1) % kUnit;
                    } else if (lane == 0) {
                        atomicOr(a.status, PKV_STATUS_BAD_SLOT);
                    }
                }
            }
        }

        __syncwarp();  // the previous run's query fragments are no longer read
        const QShared qs{stage_query<T, D>(a, b, kvh, g, c, &sm_q[warp][0][lane])};
        WarpState<MT> ws;
        ws.m0 = ws.m1 = neg_inf();
        ws.l0 = ws.l1 = 0.f;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) ws.o[mt][0] = ws.o[mt][1] = ws.o[mt][2] = ws.o[mt][3] = 0.f;

        // the appended unit is the run's last: attended after the loop
        UnitIds<BS> tab;
        tab.e0 = tab.e1 = 0;
        int k = 0, lb = lb0;
        for (; lb < lb1 && lb != app_lb; ++k, ++lb) {
            if ((k & 31) == 0) {  // table entries of the next 32 units of the run
                const int idx = lb + lane;
                tab.load(trow, idx, idx < lb1, nent);
            }
            const UnitIds<BS> e = tab.shfl(k & 31);
            if (!e.valid(a.num_blocks)) {
                if (lane == 0) atomicOr(a.status, PKV_STATUS_BAD_BLOCK);
                continue;
            }
            int64_t lo, hi;
            e.template bases<D>(a.hkv, kvh, lb, lo, hi);
            attend_block<T, D, false>(a, b, kvh, lb, lo, hi, ctx, 0, qs, ws, g, c);
        }
        if constexpr (APPEND) {
            if (lb == app_lb) attend_appended<T, D, BS>(a, b, kvh, lb, trow, nent, ctx, app_off, qs, ws, g, c);
        }

        float l0 = ws.l0, l1 = ws.l1;
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            l0 += __shfl_xor_sync(0xffffffffu, l0, off);
            l1 += __shfl_xor_sync(0xffffffffu, l1, off);
        }
        // partial (m, l, o) of this run: o staged through shared memory so
        // the G x D rows go out in 16-byte stores
        __syncwarp();
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            const int dl = pv_col(mt, g), dh = pv_col(mt + D / 16, g);
            sm_o[warp][2 * c][dl] = ws.o[mt][0];
            sm_o[warp][2 * c + 1][dl] = ws.o[mt][1];
            sm_o[warp][2 * c][dh] = ws.o[mt][2];
            sm_o[warp][2 * c + 1][dh] = ws.o[mt][3];
        }
        __syncwarp();
        const int64_t slot = i + b * a.hkv + kvh;
        float4* po = reinterpret_cast<float4*>(a.ws_o + slot * a.G * D);
        const float4* so = reinterpret_cast<const float4*>(&sm_o[warp][0][0]);
        for (int x = lane; x < a.G * D / 4; x += 32) po[x] = so[x];
        if (g == 0) {
            float* pml = a.ws_ml + slot * a.G * 2;
            if (2 * c < a.G) {
                pml[4 * c] = ws.m0;
                pml[4 * c + 1] = l0;
            }
            if (2 * c + 1 < a.G) {
                pml[4 * c + 2] = ws.m1;
                pml[4 * c + 3] = l1;
            }
        }
    }
}

// Merge of a balanced split for one (sequence, query head): the partials of
// the consecutive warps whose ranges met the (sequence, KV head) run, folded
// as in merge_kernel.  Launched behind the balanced kernel with programmatic
// dependent launch.
template <typename T, int D, int PG>
__global__ void __launch_bounds__(D * PG) merge_balanced_kernel(
    const int32_t* __restrict__ ctx_lens, int batch, int hq, int hkv, int cap,
    int nwt_launch, int min_items, const float* __restrict__ ws_o,
    const float* __restrict__ ws_ml, T* __restrict__ out) {
    constexpr int NT = D * PG, NWARP = NT / 32;
    const int h = blockIdx.x, b = blockIdx.y;
    const int d = threadIdx.x % D, pg = threadIdx.x / D;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int G = hq / hkv, kvh = h / G, hl = h - kvh * G;
    // Where the run sits among the items follows from the context lengths
    // alone -- inputs of the call, not outputs of the decode grid -- so it is
    // worked out before the wait: the blocks of the sequences before b and
    // of all sequences.
    int before = 0, total = 0;
    for (int j = threadIdx.x; j < batch; j += NT) {
        const int nbj = blocks_of(ctx_lens[j], cap);
        total += nbj;
        before += j < b ? nbj : 0;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        total += __shfl_xor_sync(0xffffffffu, total, off);
        before += __shfl_xor_sync(0xffffffffu, before, off);
    }
    __shared__ int red[2][NWARP];
    if (lane == 0) {
        red[0][warp] = total;
        red[1][warp] = before;
    }
    __syncthreads();
    total = before = 0;
#pragma unroll
    for (int w = 0; w < NWARP; ++w) {
        total += red[0][w];
        before += red[1][w];
    }
    const int nb = blocks_of(ctx_lens[b], cap);
    T* o = out + (static_cast<int64_t>(b) * hq + h) * D + d;
    // partials are produced by the preceding grid: wait for it
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (nb == 0) {
        if (pg == 0) *o = Half16<T>::from_float(0.f);
        return;
    }
    const int W = total * hkv;
    const int nwt = max(min(W / min_items, nwt_launch), 1);
    const int S = before * hkv + kvh * nb;
    const int64_t i0 = first_warp(S, W, nwt), i1 = first_warp(S + nb - 1, W, nwt);
    const int np = static_cast<int>(i1 - i0 + 1);
    const int64_t slot0 = i0 + static_cast<int64_t>(b) * hkv + kvh;
    const MergeAcc r = merge_range(ws_ml + (slot0 * G + hl) * 2, 2 * G, ws_o + (slot0 * G + hl) * D + d,
                                   static_cast<int64_t>(G) * D, pg, np, PG);
    if constexpr (PG == 1) {
        *o = Half16<T>::from_float(r.L > 0.f ? r.acc / r.L : 0.f);
        return;
    }
    __shared__ float sm[3][PG][D];
    sm[0][pg][d] = r.M;
    sm[1][pg][d] = r.L;
    sm[2][pg][d] = r.acc;
    __syncthreads();
    if (pg == 0) {
        float M = neg_inf();
#pragma unroll
        for (int j = 0; j < PG; ++j) M = fmaxf(M, sm[0][j][d]);
        float L = 0.f, acc = 0.f;
        if (M != neg_inf()) {
#pragma unroll
            for (int j = 0; j < PG; ++j) {
                const float w = ex2(sm[0][j][d] - M);
                L += w * sm[1][j][d];
                acc += w * sm[2][j][d];
            }
        }
        *o = Half16<T>::from_float(L > 0.f ? acc / L : 0.f);
    }
}

// Merge the partition partials of one (sequence, query head).  CTA of
// D x PG threads: thread (group pg, column d) folds partitions pg, pg + PG,
// ...; the PG running triples are then combined through shared memory.
// PG = 1 for up to 16 partitions, 4 beyond (long contexts).  Launched right
// behind the partition kernel with programmatic dependent launch (see
// launch_merge).
template <typename T, int D, int PG>
__global__ void __launch_bounds__(D * PG) merge_kernel(
    const int32_t* __restrict__ ctx_lens, int hq, int cap, int part_blocks, int max_parts,
    const float* __restrict__ ws_o, const float* __restrict__ ws_ml, T* __restrict__ out) {
    const int h = blockIdx.x, b = blockIdx.y;
    const int d = threadIdx.x % D, pg = threadIdx.x / D;
    int ctx = ctx_lens[b];
    ctx = ctx < 0 ? 0 : (ctx > cap ? cap : ctx);
    const int nblk = (ctx + kUnit - 1) / kUnit;  // units
    const int np = (nblk + part_blocks - 1) / part_blocks;
    const int64_t row0 = (static_cast<int64_t>(b) * hq + h) * max_parts;
    // partials are produced by the preceding grid: wait for it (a no-op
    // when this grid was launched without programmatic serialization)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const MergeAcc r = merge_range(ws_ml + 2 * row0, 2, ws_o + row0 * D + d, D, pg, np, PG);
    if constexpr (PG == 1) {
        out[(static_cast<int64_t>(b) * hq + h) * D + d] =
            Half16<T>::from_float(r.L > 0.f ? r.acc / r.L : 0.f);
        return;
    }
    __shared__ float sm[3][PG][D];
    sm[0][pg][d] = r.M;
    sm[1][pg][d] = r.L;
    sm[2][pg][d] = r.acc;
    __syncthreads();
    if (pg == 0) {
        float M = neg_inf();
#pragma unroll
        for (int j = 0; j < PG; ++j) M = fmaxf(M, sm[0][j][d]);
        float L = 0.f, acc = 0.f;
        if (M != neg_inf()) {
#pragma unroll
            for (int j = 0; j < PG; ++j) {
                const float w = ex2(sm[0][j][d] - M);
                L += w * sm[1][j][d];
                acc += w * sm[2][j][d];
            }
        }
        out[(static_cast<int64_t>(b) * hq + h) * D + d] = Half16<T>::from_float(L > 0.f ? acc / L : 0.f);
    }
}

// part_blocks: 16-token units per partition; units: units per table.
struct Shape {
    int batch, hq, hkv, D, num_blocks, block_size, max_blocks, part_blocks, max_parts;
    int cap, units;  // table capacity in tokens and in 16-token units
    bool balanced;   // automatic split: balanced over warps instead of fixed partitions
};


}  // namespace

// SM count of the current device (152 when it cannot be queried), cached.
int num_sms() {
    static std::atomic<int> sms{0};
    int n = sms.load();
    if (n == 0) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 152;
        sms.store(n);
    }
    return n;
}

// Automatic partition size: the largest of 512, 256, 128, 64 tokens that
// still gives >= 12 x SMs (query head, partition) work items, i.e. ~3
// partition CTAs per SM at a GQA group of 4; small batches get finer splits.
// (Measured on the 8-sequence prefix workload: 256 beat both 128 and 512.)
int auto_partition_size(int32_t batch, int32_t hq, int64_t tokens) {
    const int n = num_sms();
    for (int ps = 512; ps > 64; ps /= 2) {
        const int64_t parts = (tokens + ps - 1) / ps;
        if (static_cast<int64_t>(batch) * hq * parts >= 12LL * n) return ps;
    }
    return 64;
}

// No more warps than the largest possible item count allows at
// kBalancedMinItems each, so small problems launch (and need room for) fewer.
int balanced_warps(int64_t max_items, int warps_per_sm) {
    const int64_t full = static_cast<int64_t>(num_sms()) * warps_per_sm;
    const int64_t n = max_items / kBalancedMinItems < full ? max_items / kBalancedMinItems : full;
    return n < 1 ? 1 : static_cast<int>(n);
}

bool balanced_candidate(int64_t batch, int64_t max_items) {
    return batch <= kBalancedMaxBatch &&
           max_items >= static_cast<int64_t>(kBalancedItemsPerWarp) * num_sms() * 16;
}

bool use_balanced(int64_t batch, int64_t hkv, int64_t max_units) {
    const int64_t items = batch * hkv * max_units;
    return balanced_candidate(batch, items) && items < (1LL << 30);
}

size_t balanced_bytes(int32_t batch, int32_t hq, int32_t G, int32_t D, int32_t nwt) {
    const size_t rows = static_cast<size_t>(nwt) * G + static_cast<size_t>(batch) * hq;
    return rows * (D + 2) * sizeof(float);
}

namespace {

// Block sizes the 16-bit decode kernels are built for.
bool block_size_supported(int32_t bs) { return bs == 8 || bs == 16 || bs == 32; }

// Partition layout of a split-K call: units per table, 16-token units per
// partition and partitions per table.  partition_size (0: automatic) must be
// a positive multiple of both 16 and block_size.
int partition_layout(int32_t batch, int32_t hq, int32_t max_blocks, int32_t block_size,
                     int32_t partition_size, Shape* s) {
    const int64_t cap = static_cast<int64_t>(max_blocks) * block_size;
    if (cap > (1LL << 30)) return PKV_ERR_UNSUPPORTED;
    if (partition_size == 0) partition_size = auto_partition_size(batch, hq, cap);
    if (partition_size % block_size != 0 || partition_size % kUnit != 0) return PKV_ERR_INVALID_ARG;
    s->cap = static_cast<int>(cap);
    s->units = static_cast<int>((cap + kUnit - 1) / kUnit);
    s->part_blocks = partition_size / kUnit;
    s->max_parts = (s->units + s->part_blocks - 1) / s->part_blocks;
    if (s->max_parts < 1) s->max_parts = 1;
    return PKV_OK;
}

int check_shape(int32_t batch, int32_t hq, int32_t hkv, int32_t D, int32_t num_blocks,
                int32_t block_size, int32_t max_blocks, int32_t partition_size, int dtype,
                Shape* s) {
    if (batch < 0 || hq <= 0 || hkv <= 0 || D <= 0 || num_blocks <= 0 || block_size <= 0 ||
        max_blocks < 0 || partition_size < 0)
        return PKV_ERR_INVALID_ARG;
    if (dtype != PKV_DTYPE_F16 && dtype != PKV_DTYPE_BF16) return PKV_ERR_INVALID_ARG;
    if (hq % hkv != 0) return PKV_ERR_INVALID_ARG;
    if (!block_size_supported(block_size) || (D != 64 && D != 128) || hq / hkv > 8)
        return PKV_ERR_UNSUPPORTED;
    if (batch > 65535 || hkv > 65535) return PKV_ERR_UNSUPPORTED;
    const int st = partition_layout(batch, hq, max_blocks, block_size, partition_size, s);
    if (st != PKV_OK) return st;
    s->balanced = partition_size == 0 && use_balanced(batch, hkv, s->units);
    s->batch = batch;
    s->hq = hq;
    s->hkv = hkv;
    s->D = D;
    s->num_blocks = num_blocks;
    s->block_size = block_size;
    s->max_blocks = max_blocks;
    return PKV_OK;
}

size_t partial_bytes(const Shape& s) {
    return static_cast<size_t>(s.batch) * s.hq * s.max_parts * (s.D + 2) * sizeof(float);
}

template <typename T, int D, int MODE, bool APPEND, int BS>
int launch_kernel(const DecodeArgs& a, const Shape& s, cudaStream_t st) {
    dim3 grid(MODE == kSingle ? 1 : s.max_parts, s.hkv, s.batch);
    paged_decode_kernel<T, D, kNW, MODE, APPEND, BS><<<grid, kNW * 32, 0, st>>>(a);
    return launch_status();
}

template <int MODE, bool APPEND, int BS>
int dispatch_bs(const DecodeArgs& a, const Shape& s, int dtype, cudaStream_t st) {
    if (dtype == PKV_DTYPE_BF16) {
        if (s.D == 128) return launch_kernel<__nv_bfloat16, 128, MODE, APPEND, BS>(a, s, st);
        return launch_kernel<__nv_bfloat16, 64, MODE, APPEND, BS>(a, s, st);
    }
    if (s.D == 128) return launch_kernel<__half, 128, MODE, APPEND, BS>(a, s, st);
    return launch_kernel<__half, 64, MODE, APPEND, BS>(a, s, st);
}

template <int MODE, bool APPEND>
int dispatch(const DecodeArgs& a, const Shape& s, int dtype, cudaStream_t st) {
    if (s.block_size == 8) return dispatch_bs<MODE, APPEND, 8>(a, s, dtype, st);
    if (s.block_size == 32) return dispatch_bs<MODE, APPEND, 32>(a, s, dtype, st);
    return dispatch_bs<MODE, APPEND, 16>(a, s, dtype, st);
}

template <typename T, int D, int PG>
int launch_merge_balanced_t(const int32_t* ctx_lens, int batch, int hq, int hkv, int cap, int nwt,
                            const float* ws_o, const float* ws_ml, void* out, cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(hq, batch);
    cfg.blockDim = dim3(D * PG);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, merge_balanced_kernel<T, D, PG>, ctx_lens, batch, hq, hkv,
                                             cap, nwt, kBalancedMinItems, ws_o, ws_ml,
                                             static_cast<T*>(out));
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

// Balanced split: the warp-range kernel, then its merge.
template <typename T, int D, bool APPEND, int BS>
int run_balanced(const DecodeArgs& a, const Shape& s, int nwt, cudaStream_t st) {
    paged_decode_balanced_kernel<T, D, APPEND, BS>
        <<<(nwt + kNW - 1) / kNW, kNW * 32, 0, st>>>(a, s.batch, nwt, kBalancedMinItems);
    const int r = launch_status();
    if (r != PKV_OK) return r;
    return launch_balanced_merge(a.ctx_lens, s.batch, s.hq, s.hkv, D, s.cap, nwt, a.ws_o, a.ws_ml, a.out,
                                 std::is_same<T, __half>::value ? PKV_DTYPE_F16 : PKV_DTYPE_BF16, st);
}

template <bool APPEND, int BS>
int dispatch_balanced_bs(const DecodeArgs& a, const Shape& s, int nwt, int dtype, cudaStream_t st) {
    if (dtype == PKV_DTYPE_BF16) {
        if (s.D == 128) return run_balanced<__nv_bfloat16, 128, APPEND, BS>(a, s, nwt, st);
        return run_balanced<__nv_bfloat16, 64, APPEND, BS>(a, s, nwt, st);
    }
    if (s.D == 128) return run_balanced<__half, 128, APPEND, BS>(a, s, nwt, st);
    return run_balanced<__half, 64, APPEND, BS>(a, s, nwt, st);
}

template <bool APPEND>
int dispatch_balanced(const DecodeArgs& a, const Shape& s, int nwt, int dtype, cudaStream_t st) {
    if (s.block_size == 8) return dispatch_balanced_bs<APPEND, 8>(a, s, nwt, dtype, st);
    if (s.block_size == 32) return dispatch_balanced_bs<APPEND, 32>(a, s, nwt, dtype, st);
    return dispatch_balanced_bs<APPEND, 16>(a, s, nwt, dtype, st);
}

// The merge grid is launched with programmatic stream serialization: it may
// be scheduled as soon as every CTA of the preceding grid has started, and
// its griddepcontrol.wait holds each CTA until that grid has completed and
// its writes are visible.  This hides the second launch behind the first
// grid's last wave.
template <typename T, int D, int PG>
int launch_merge(const int32_t* ctx_lens, const Shape& s, const float* ws_o, const float* ws_ml,
                 void* out, cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(s.hq, s.batch);
    cfg.blockDim = dim3(D * PG);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, merge_kernel<T, D, PG>, ctx_lens, s.hq, s.cap,
                                             s.part_blocks, s.max_parts, ws_o, ws_ml,
                                             static_cast<T*>(out));
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

int run_merge(const int32_t* ctx_lens, const Shape& s, const float* ws_o, const float* ws_ml,
              void* out, int dtype, cudaStream_t st) {
    const bool many = s.max_parts > 16;
#define PKV_MERGE(TT, DD)                                                                       \
    return many ? launch_merge<TT, DD, 4>(ctx_lens, s, ws_o, ws_ml, out, st)                   \
                : launch_merge<TT, DD, 1>(ctx_lens, s, ws_o, ws_ml, out, st)
    if (dtype == PKV_DTYPE_BF16) {
        if (s.D == 128) PKV_MERGE(__nv_bfloat16, 128);
        PKV_MERGE(__nv_bfloat16, 64);
    }
    if (s.D == 128) PKV_MERGE(__half, 128);
    PKV_MERGE(__half, 64);
#undef PKV_MERGE
}

int fill_args(DecodeArgs* a, const void* q, const void* k_pool, const void* v_pool,
              const int32_t* tables, const int32_t* ctx_lens, const Shape& s, float scale) {
    if (!q || !k_pool || !v_pool || !tables || !ctx_lens) return PKV_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) ||
        (reinterpret_cast<uintptr_t>(tables) & 3u) || (reinterpret_cast<uintptr_t>(ctx_lens) & 3u))
        return PKV_ERR_MISALIGNED;
    int* st = status_word();
    if (!st) return PKV_ERR_CUDA;
    *a = DecodeArgs{};
    a->q = q;
    a->k_pool = k_pool;
    a->v_pool = v_pool;
    a->tables = tables;
    a->ctx_lens = ctx_lens;
    a->hq = s.hq;
    a->hkv = s.hkv;
    a->G = s.hq / s.hkv;
    a->num_blocks = s.num_blocks;
    a->max_blocks = s.max_blocks;
    a->cap = s.cap;
    a->part_blocks = s.part_blocks;
    a->max_parts = s.max_parts;
    a->scale_log2 = scale * kLog2e;
    a->status = st;
    return PKV_OK;
}

int set_workspace(DecodeArgs* a, const Shape& s, void* ws, size_t bytes) {
    if (!ws || bytes < partial_bytes(s)) return PKV_ERR_WORKSPACE;
    if (!aligned16(ws)) return PKV_ERR_MISALIGNED;
    a->ws_o = static_cast<float*>(ws);
    a->ws_ml = a->ws_o + static_cast<size_t>(s.batch) * s.hq * s.max_parts * s.D;
    return PKV_OK;
}

// One decode call: single pass when one partition covers every table;
// otherwise, with the automatic split, the balanced kernel then its merge,
// else the partition kernel then the merge kernel.
template <bool APPEND>
int decode(const DecodeArgs& a0, const Shape& s, void* out, void* ws, size_t ws_bytes, int dtype,
           cudaStream_t cs) {
    DecodeArgs a = a0;
    a.out = out;
    if (s.max_parts <= 1) {
        a.part_blocks = s.units > 0 ? s.units : 1;
        return dispatch<kSingle, APPEND>(a, s, dtype, cs);
    }
    if (s.balanced) {
        // 4 CTAs of 4 warps per SM
        const int nwt = balanced_warps(static_cast<int64_t>(s.batch) * s.hkv * s.units, 4 * kNW);
        const int G = s.hq / s.hkv;
        if (!ws || ws_bytes < balanced_bytes(s.batch, s.hq, G, s.D, nwt)) return PKV_ERR_WORKSPACE;
        if (!aligned16(ws)) return PKV_ERR_MISALIGNED;
        const size_t rows = static_cast<size_t>(nwt) * G + static_cast<size_t>(s.batch) * s.hq;
        a.ws_o = static_cast<float*>(ws);
        a.ws_ml = a.ws_o + rows * s.D;
        return dispatch_balanced<APPEND>(a, s, nwt, dtype, cs);
    }
    int st = set_workspace(&a, s, ws, ws_bytes);
    if (st != PKV_OK) return st;
    if ((st = dispatch<kPartials, APPEND>(a, s, dtype, cs)) != PKV_OK) return st;
    return run_merge(a.ctx_lens, s, a.ws_o, a.ws_ml, out, dtype, cs);
}

}  // namespace

// Runs of one (sequence, KV head) span about nwt / (batch * Hkv) warp ranges
// at the longest; beyond 16 the merge folds with 4 partial groups per CTA.
int launch_balanced_merge(const int32_t* ctx_lens, int batch, int hq, int hkv, int D, int cap, int nwt,
                          const float* ws_o, const float* ws_ml, void* out, int dtype, cudaStream_t st) {
    const bool many = nwt > 16LL * batch * hkv;
#define PKV_BMERGE(TT, DD)                                                                                \
    return many ? launch_merge_balanced_t<TT, DD, 4>(ctx_lens, batch, hq, hkv, cap, nwt, ws_o, ws_ml, out, \
                                                     st)                                                  \
                : launch_merge_balanced_t<TT, DD, 1>(ctx_lens, batch, hq, hkv, cap, nwt, ws_o, ws_ml, out, st)
    if (dtype == PKV_DTYPE_BF16) {
        if (D == 128) PKV_BMERGE(__nv_bfloat16, 128);
        PKV_BMERGE(__nv_bfloat16, 64);
    }
    if (D == 128) PKV_BMERGE(__half, 128);
    PKV_BMERGE(__half, 64);
#undef PKV_BMERGE
}

}  // namespace pkv

extern "C" int pkv_decode_workspace_bytes(int32_t batch, int32_t num_q_heads, int32_t head_dim,
                                          int32_t max_blocks, int32_t block_size,
                                          int32_t partition_size, size_t* out) {
    if (!out || batch < 0 || num_q_heads <= 0 || head_dim <= 0 || max_blocks < 0 ||
        block_size <= 0 || partition_size < 0)
        return PKV_ERR_INVALID_ARG;
    const bool automatic = partition_size == 0;
    pkv::Shape s;
    const int st = pkv::partition_layout(batch, num_q_heads, max_blocks, block_size, partition_size, &s);
    if (st != PKV_OK) return st;
    const int64_t parts = s.max_parts;
    if (parts <= 1) {
        *out = 0;
        return PKV_OK;
    }
    const size_t fixed = static_cast<size_t>(batch) * num_q_heads * parts * (head_dim + 2) * sizeof(float);
    const int64_t max_items = static_cast<int64_t>(batch) * num_q_heads * s.units;  // Hkv <= Hq
    if (automatic && pkv::balanced_candidate(batch, max_items)) {
        // room for a balanced split (16-bit cache) with Hkv anywhere in
        // [1, Hq] and a GQA group up to 8; the quantised decode still splits
        // into the automatic partitions
        const int nwt = pkv::balanced_warps(max_items, pkv::kBalancedMaxWarpsPerSm);
        const size_t bal = pkv::balanced_bytes(batch, num_q_heads, 8, head_dim, nwt);
        *out = bal > fixed ? bal : fixed;
        return PKV_OK;
    }
    *out = fixed;
    return PKV_OK;
}

extern "C" int pkv_paged_attention_decode_partials(
    const void* q, const void* k_pool, const void* v_pool, const int32_t* block_tables,
    const int32_t* context_lens, int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
    int32_t head_dim, int32_t num_blocks, int32_t block_size, int32_t max_blocks, float scale,
    void* workspace, size_t workspace_bytes, int32_t partition_size, int dtype, void* stream) {
    pkv::Shape s;
    int st = pkv::check_shape(batch, num_q_heads, num_kv_heads, head_dim, num_blocks, block_size,
                              max_blocks, partition_size, dtype, &s);
    if (st != PKV_OK) return st;
    if (batch == 0 || max_blocks == 0) return PKV_OK;
    pkv::DecodeArgs a;
    if ((st = pkv::fill_args(&a, q, k_pool, v_pool, block_tables, context_lens, s, scale)) != PKV_OK)
        return st;
    if ((st = pkv::set_workspace(&a, s, workspace, workspace_bytes)) != PKV_OK) return st;
    pkv::dispatch<pkv::kPartials, false>(a, s, dtype, static_cast<cudaStream_t>(stream));
    return pkv::launch_status();
}

extern "C" int pkv_paged_attention_decode_merge(const int32_t* context_lens, int32_t batch,
                                                int32_t num_q_heads, int32_t head_dim,
                                                int32_t max_blocks, int32_t block_size,
                                                int32_t partition_size, const void* workspace,
                                                size_t workspace_bytes, void* out, int dtype,
                                                void* stream) {
    // The merge never reads the pool, so only the partial-buffer shape matters.
    if (batch < 0 || num_q_heads <= 0 || max_blocks < 0 || partition_size < 0 ||
        (dtype != PKV_DTYPE_F16 && dtype != PKV_DTYPE_BF16))
        return PKV_ERR_INVALID_ARG;
    if (!pkv::block_size_supported(block_size) || (head_dim != 64 && head_dim != 128) || batch > 65535 ||
        num_q_heads > 65535)
        return PKV_ERR_UNSUPPORTED;
    pkv::Shape s;
    const int st = pkv::partition_layout(batch, num_q_heads, max_blocks, block_size, partition_size, &s);
    if (st != PKV_OK) return st;
    s.batch = batch;
    s.hq = num_q_heads;
    s.hkv = 1;
    s.D = head_dim;
    s.num_blocks = 1;
    s.block_size = block_size;
    s.max_blocks = max_blocks;
    s.balanced = false;
    if (batch == 0) return PKV_OK;
    if (!context_lens || !out) return PKV_ERR_INVALID_ARG;
    if (!pkv::aligned16(out)) return PKV_ERR_MISALIGNED;
    if (!workspace || workspace_bytes < pkv::partial_bytes(s)) return PKV_ERR_WORKSPACE;
    if (!pkv::aligned16(workspace)) return PKV_ERR_MISALIGNED;
    const float* ws_o = static_cast<const float*>(workspace);
    const float* ws_ml = ws_o + static_cast<size_t>(s.batch) * s.hq * s.max_parts * s.D;
    return pkv::run_merge(context_lens, s, ws_o, ws_ml, out, dtype, static_cast<cudaStream_t>(stream));
}

extern "C" int pkv_paged_attention_decode(const void* q, const void* k_pool, const void* v_pool,
                                          const int32_t* block_tables, const int32_t* context_lens,
                                          int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                          int32_t head_dim, int32_t num_blocks, int32_t block_size,
                                          int32_t max_blocks, float scale, void* out,
                                          void* workspace, size_t workspace_bytes,
                                          int32_t partition_size, int dtype, void* stream) {
    pkv::Shape s;
    int st = pkv::check_shape(batch, num_q_heads, num_kv_heads, head_dim, num_blocks, block_size,
                              max_blocks, partition_size, dtype, &s);
    if (st != PKV_OK) return st;
    if (batch == 0) return PKV_OK;
    if (!out) return PKV_ERR_INVALID_ARG;
    if (!pkv::aligned16(out)) return PKV_ERR_MISALIGNED;
    pkv::DecodeArgs a;
    if ((st = pkv::fill_args(&a, q, k_pool, v_pool, block_tables, context_lens, s, scale)) != PKV_OK)
        return st;
    return pkv::decode<false>(a, s, out, workspace, workspace_bytes, dtype,
                              static_cast<cudaStream_t>(stream));
}

extern "C" int pkv_paged_attention_decode_append(
    const void* q, const void* k_new, const void* v_new, const int64_t* slot_mapping,
    void* k_pool, void* v_pool, const int32_t* block_tables, const int32_t* context_lens,
    int32_t batch, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
    int32_t num_blocks, int32_t block_size, int32_t max_blocks, float scale, void* out,
    void* workspace, size_t workspace_bytes, int32_t partition_size, int dtype, void* stream) {
    pkv::Shape s;
    int st = pkv::check_shape(batch, num_q_heads, num_kv_heads, head_dim, num_blocks, block_size,
                              max_blocks, partition_size, dtype, &s);
    if (st != PKV_OK) return st;
    if (batch == 0) return PKV_OK;
    if (!out || !k_new || !v_new || !slot_mapping) return PKV_ERR_INVALID_ARG;
    if (!pkv::aligned16(out) || !pkv::aligned16(k_new) || !pkv::aligned16(v_new) ||
        (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
        return PKV_ERR_MISALIGNED;
    pkv::DecodeArgs a;
    if ((st = pkv::fill_args(&a, q, k_pool, v_pool, block_tables, context_lens, s, scale)) != PKV_OK)
        return st;
    a.k_pool_w = k_pool;
    a.v_pool_w = v_pool;
    a.k_new = k_new;
    a.v_new = v_new;
    a.slots = slot_mapping;
    return pkv::decode<true>(a, s, out, workspace, workspace_bytes, dtype,
                             static_cast<cudaStream_t>(stream));
}

extern "C" int pkv_decode_auto_partition_size(int32_t batch, int32_t num_q_heads, int32_t max_blocks,
                                              int32_t block_size, int32_t* out) {
    if (!out || batch < 0 || num_q_heads <= 0 || max_blocks < 0) return PKV_ERR_INVALID_ARG;
    if (!pkv::block_size_supported(block_size)) return PKV_ERR_UNSUPPORTED;
    *out = pkv::auto_partition_size(batch, num_q_heads, static_cast<int64_t>(max_blocks) * block_size);
    return PKV_OK;
}
