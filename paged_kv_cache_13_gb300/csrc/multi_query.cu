// Multi-query paged attention: several new query tokens per sequence, each
// attending causally to the cache up to its own position.
//
// What it computes: sequence b holds ctx_b tokens in the pool (its block
// table), the last L_b of which are this call's new tokens, at positions
// ctx_b - L_b .. ctx_b - 1.  Query token i of b (row q_start[b] + i of q)
// sits at position p = ctx_b - L_b + i and
//   out[q_start[b] + i, h] = sum_{t <= p} softmax_t(scale <q, K_t>) V_t
// with K_t, V_t of KV head h / G gathered through the table.  This is the
// attention of the target model's one parallel pass over the gamma + 1
// draft tokens of speculative decoding ("The 8GB VRAM Breakthrough", §6
// "Speculative Decoding: Breaking the Bandwidth Wall") and of a 512-token
// chunk of a chunked prefill (§5, "Chunked Prefill"); with L_b = 1 it is the
// decode attention of decode.cu.
//
// Design: the layout of the decode kernels -- K and V fragments loaded
// straight from the pool into mma.sync registers, tokens as M of QK^T and
// the head dim as M of PV -- with the N dimension holding (query token,
// query head) rows instead of heads: a CTA takes a tile of 8 NT rows of one
// (sequence, KV head), NT n-tiles of 8, so every K/V fragment loaded is used
// by all rows of the tile.  Its 4 warps take the blocks up to the tile's
// last position round-robin, each with its own online softmax per row, and
// merge through shared memory.  Rows beyond a token's position are masked
// per element; blocks past the tile's last position are not read.

#include "balanced.cuh"
#include "prefill_tc.cuh"

namespace pkv {
namespace {

constexpr int BS = 16;
constexpr int NW = 4;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kSlack = 8.f;  // see the softmax in attend()

struct MQArgs {
    const void* q;
    const int32_t* q_start;
    const void* k_pool;
    const void* v_pool;
    const int32_t* tables;
    const int32_t* ctx_lens;
    int hq, hkv, G, num_blocks, max_blocks;
    float scale_log2;
    void* out;
    int* status;
};

template <typename T>
constexpr bool kSplitP = false;
template <>
constexpr bool kSplitP<__nv_bfloat16> = true;

__device__ __forceinline__ float lo_float(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float hi_float(uint32_t x) { return __uint_as_float(x & 0xffff0000u); }

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 r;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "r"(addr));
    return r;
}

// Element e (0 .. D/8-1) of lane group g in the PV fragment layout sits at
// head-dim column 64 * (e / 8) + 8 * g + e % 8.
__device__ __forceinline__ int pv_col(int e, int g) { return 64 * (e >> 3) + 8 * g + (e & 7); }

// Online-softmax state of one warp: lane (g, c) holds rows 8 nt + 2c and
// 8 nt + 2c + 1 of every n-tile nt.
template <int MT, int NT>
struct MQState {
    float m[NT][2], l[NT][2];
    float o[MT][NT][4];
};

// Attend one 16-token block (physical id phys, logical index lb).  qs: the
// lane's shared address of the tile's query fragments (n-tile nt, k-chunk i
// at qs + (nt * KC + i) * 512); pos: the positions of the lane's rows (-1
// for rows beyond the sequence's tokens).
template <typename T, int D, int NT>
__device__ __forceinline__ void attend(const MQArgs& a, int kvh, int lb, int phys, int ctx, uint32_t qs,
                                       const int (&pos)[NT][2], MQState<D / 16, NT>& w, int g, int c) {
    using H = Half16<T>;
    constexpr int KC = D / 32;
    constexpr int VC = D / 64;
    constexpr int MT = D / 16;
    const int64_t base = (static_cast<int64_t>(phys) * a.hkv + kvh) * (BS * D);
    const T* kb = static_cast<const T*>(a.k_pool) + base;
    const T* vb = static_cast<const T*>(a.v_pool) + base;

    // K rows g, g + 8 at [32i + 8c, +8); V rows 2c, 2c+1, 8+2c, 9+2c at [64j + 8g, +8)
    uint4 kr0[KC], kr1[KC], vr[4][VC];
#pragma unroll
    for (int i = 0; i < KC; ++i) {
        kr0[i] = ldg_stream(kb + g * D + 32 * i + 8 * c);
        kr1[i] = ldg_stream(kb + (g + 8) * D + 32 * i + 8 * c);
    }
#pragma unroll
    for (int j = 0; j < VC; ++j) {
        vr[0][j] = ldg_stream(vb + (2 * c) * D + 64 * j + 8 * g);
        vr[1][j] = ldg_stream(vb + (2 * c + 1) * D + 64 * j + 8 * g);
        vr[2][j] = ldg_stream(vb + (8 + 2 * c) * D + 64 * j + 8 * g);
        vr[3][j] = ldg_stream(vb + (9 + 2 * c) * D + 64 * j + 8 * g);
    }

    const int tok0 = lb * BS + g, tok1 = tok0 + 8;
    uint32_t pb0[NT], pb1[NT], pr0[NT], pr1[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        // ---- S^T = K Q^T for the 8 rows of n-tile nt (permuted k order)
        float s[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < KC; ++i) {
            const uint4 qf = lds128(qs + (nt * KC + i) * 512);
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                H::mma(s, word(kr0[i], 2 * e), word(kr1[i], 2 * e), word(kr0[i], 2 * e + 1),
                       word(kr1[i], 2 * e + 1), word(qf, 2 * e), word(qf, 2 * e + 1));
            }
        }
        // causal mask: token t is seen by a row at position p >= t
        const float x0 = tok0 <= pos[nt][0] ? s[0] * a.scale_log2 : neg_inf();
        const float x1 = tok0 <= pos[nt][1] ? s[1] * a.scale_log2 : neg_inf();
        const float x2 = tok1 <= pos[nt][0] ? s[2] * a.scale_log2 : neg_inf();
        const float x3 = tok1 <= pos[nt][1] ? s[3] * a.scale_log2 : neg_inf();

        // ---- online softmax (base 2), rows 2c (x0, x2) and 2c + 1 (x1, x3):
        // the reference max is raised only when a logit exceeds it by more
        // than kSlack (weights then stay <= 2^kSlack); otherwise no warp-wide
        // max and no rescale.
        const float bx0 = fmaxf(x0, x2), bx1 = fmaxf(x1, x3);
        if (__any_sync(0xffffffffu, bx0 > w.m[nt][0] + kSlack || bx1 > w.m[nt][1] + kSlack)) {
            float bm0 = bx0, bm1 = bx1;
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                bm0 = fmaxf(bm0, __shfl_xor_sync(0xffffffffu, bm0, off));
                bm1 = fmaxf(bm1, __shfl_xor_sync(0xffffffffu, bm1, off));
            }
            const float mn0 = fmaxf(w.m[nt][0], bm0), mn1 = fmaxf(w.m[nt][1], bm1);
            // a row still without any visible token keeps m = -inf
            const float al0 = mn0 == neg_inf() ? 1.f : ex2(w.m[nt][0] - mn0);
            const float al1 = mn1 == neg_inf() ? 1.f : ex2(w.m[nt][1] - mn1);
            w.l[nt][0] *= al0;
            w.l[nt][1] *= al1;
            w.m[nt][0] = mn0;
            w.m[nt][1] = mn1;
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                w.o[mt][nt][0] *= al0;
                w.o[mt][nt][1] *= al1;
                w.o[mt][nt][2] *= al0;
                w.o[mt][nt][3] *= al1;
            }
        }
        // masked logits give 0 even while the row's m is still -inf
        const float r0 = w.m[nt][0] == neg_inf() ? 0.f : w.m[nt][0];
        const float r1 = w.m[nt][1] == neg_inf() ? 0.f : w.m[nt][1];
        const float p0 = ex2(x0 - r0), p1 = ex2(x1 - r1);
        const float p2 = ex2(x2 - r0), p3 = ex2(x3 - r1);
        w.l[nt][0] += p0 + p2;
        w.l[nt][1] += p1 + p3;
        // P^T B-fragments (two 8x8 transposes); bf16 P also as its residual
        const uint32_t h01 = H::pack(p0, p1), h23 = H::pack(p2, p3);
        pb0[nt] = movmatrix_trans(h01);
        pb1[nt] = movmatrix_trans(h23);
        if constexpr (kSplitP<T>) {
            pr0[nt] = movmatrix_trans(H::pack(p0 - lo_float(h01), p1 - hi_float(h01)));
            pr1[nt] = movmatrix_trans(H::pack(p2 - lo_float(h23), p3 - hi_float(h23)));
        }
    }

    // ---- O^T += V^T P^T; every V fragment serves all NT n-tiles.  Masked
    // tokens have P = 0, but slots past the context may hold any bits (NaN
    // included, and 0 * NaN would poison o): their V rows are cleared.
    if (lb * BS + BS > ctx) {
        const int t0 = lb * BS;
#pragma unroll
        for (int j = 0; j < VC; ++j) {
            if (t0 + 2 * c >= ctx) vr[0][j] = make_uint4(0, 0, 0, 0);
            if (t0 + 2 * c + 1 >= ctx) vr[1][j] = make_uint4(0, 0, 0, 0);
            if (t0 + 8 + 2 * c >= ctx) vr[2][j] = make_uint4(0, 0, 0, 0);
            if (t0 + 9 + 2 * c >= ctx) vr[3][j] = make_uint4(0, 0, 0, 0);
        }
    }
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
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            H::mma(w.o[mt][nt], a0, a1, a2, a3, pb0[nt], pb1[nt]);
            if constexpr (kSplitP<T>) H::mma(w.o[mt][nt], a0, a1, a2, a3, pr0[nt], pr1[nt]);
        }
    }
}

// One CTA per (row tile, KV head, sequence).  Row r of the tile (0 .. 8 NT - 1)
// is row tile * 8 NT + r of the sequence's (query token, query head) rows,
// token i = row / G, head kvh * G + row % G.
template <typename T, int D, int NT>
__global__ void __launch_bounds__(NW * 32, NT == 1 ? 4 : 3) multi_query_kernel(MQArgs a) {
    using H = Half16<T>;
    constexpr int KC = D / 32;
    constexpr int MT = D / 16;
    constexpr int R = 8 * NT;
    const int tile = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, c = lane & 3;

    const int q0 = a.q_start[b], L = a.q_start[b + 1] - q0;
    const int row0 = tile * R;
    if (L <= 0 || row0 >= L * a.G) return;
    int ctx = a.ctx_lens[b];
    const int cap = a.max_blocks * BS;
    if (ctx < L || ctx > cap) {
        if (threadIdx.x == 0 && tile == 0 && kvh == 0) atomicOr(a.status, PKV_STATUS_BAD_CONTEXT);
        ctx = ctx > cap ? cap : ctx;
    }
    const int first_pos = ctx - L;  // position of query token 0 (negative if ctx < L)

    // query fragments of the tile, shared by the 4 warps: n-tile nt, column g
    // (row 8 nt + g), k-chunk i at sq[nt][i][lane]
    __shared__ uint4 sq[NT][KC][32];
    for (int x = threadIdx.x; x < NT * KC * 32; x += NW * 32) {
        const int nt = x / (KC * 32), i = (x / 32) % KC, ln = x % 32;
        const int row = row0 + 8 * nt + (ln >> 2), cc = ln & 3;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (row < L * a.G) {
            const int tok = row / a.G, h = row - tok * a.G;
            const T* qrow = static_cast<const T*>(a.q) +
                            ((static_cast<int64_t>(q0) + tok) * a.hq + kvh * a.G + h) * D;
            v = *reinterpret_cast<const uint4*>(qrow + 32 * i + 8 * cc);
        }
        sq[nt][i][ln] = v;
    }
    __syncthreads();
    const uint32_t qs = static_cast<uint32_t>(__cvta_generic_to_shared(&sq[0][0][lane]));

    // positions of this lane's rows (8 nt + 2c, 8 nt + 2c + 1), -1 if none
    int pos[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int row = row0 + 8 * nt + 2 * c + k;
            const int p = row < L * a.G ? first_pos + row / a.G : -1;
            pos[nt][k] = p < 0 ? -1 : p;
        }
    }
    // blocks up to the tile's last position (its last valid row's token)
    const int last = first_pos + (min(row0 + R, L * a.G) - 1) / a.G;
    const int nblk = last >= 0 ? last / BS + 1 : 0;

    MQState<MT, NT> w;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        w.m[nt][0] = w.m[nt][1] = neg_inf();
        w.l[nt][0] = w.l[nt][1] = 0.f;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) w.o[mt][nt][0] = w.o[mt][nt][1] = w.o[mt][nt][2] = w.o[mt][nt][3] = 0.f;
    }
    const int32_t* trow = a.tables + static_cast<int64_t>(b) * a.max_blocks;
    int tab = 0, k = 0;
    for (int lb = warp; lb < nblk; lb += NW, ++k) {
        if ((k & 31) == 0) {  // physical ids of this warp's next 32 blocks
            const int idx = lb + NW * lane;
            tab = idx < nblk ? trow[idx] : 0;
        }
        const int phys = __shfl_sync(0xffffffffu, tab, k & 31);
        if (static_cast<unsigned>(phys) >= static_cast<unsigned>(a.num_blocks)) {
            if (lane == 0) atomicOr(a.status, PKV_STATUS_BAD_BLOCK);
            continue;
        }
        attend<T, D, NT>(a, kvh, lb, phys, ctx, qs, pos, w, g, c);
    }

    // ---- merge the NW warps through shared memory, write the tile's rows
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            w.l[nt][0] += __shfl_xor_sync(0xffffffffu, w.l[nt][0], off);
            w.l[nt][1] += __shfl_xor_sync(0xffffffffu, w.l[nt][1], off);
        }
    }
    __shared__ float sm_ml[NW][R][2];
    __shared__ float sm_o[NW][R][D];
    if (g == 0) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            sm_ml[warp][8 * nt + 2 * c][0] = w.m[nt][0];
            sm_ml[warp][8 * nt + 2 * c][1] = w.l[nt][0];
            sm_ml[warp][8 * nt + 2 * c + 1][0] = w.m[nt][1];
            sm_ml[warp][8 * nt + 2 * c + 1][1] = w.l[nt][1];
        }
    }
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
        const int dl = pv_col(mt, g), dh = pv_col(mt + D / 16, g);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            sm_o[warp][8 * nt + 2 * c][dl] = w.o[mt][nt][0];
            sm_o[warp][8 * nt + 2 * c + 1][dl] = w.o[mt][nt][1];
            sm_o[warp][8 * nt + 2 * c][dh] = w.o[mt][nt][2];
            sm_o[warp][8 * nt + 2 * c + 1][dh] = w.o[mt][nt][3];
        }
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < R * D; idx += NW * 32) {
        const int r = idx / D, d = idx - r * D;
        const int row = row0 + r;
        if (row >= L * a.G) continue;
        float M = neg_inf();
#pragma unroll
        for (int ww = 0; ww < NW; ++ww) M = fmaxf(M, sm_ml[ww][r][0]);
        float acc = 0.f, Ls = 0.f;
        if (M != neg_inf()) {
#pragma unroll
            for (int ww = 0; ww < NW; ++ww) {
                const float sc = ex2(sm_ml[ww][r][0] - M);
                acc += sc * sm_o[ww][r][d];
                Ls += sc * sm_ml[ww][r][1];
            }
        }
        const int tok = row / a.G, h = row - tok * a.G;
        const int64_t orow = (static_cast<int64_t>(q0) + tok) * a.hq + kvh * a.G + h;
        static_cast<T*>(a.out)[orow * D + d] = H::from_float(Ls > 0.f ? acc / Ls : 0.f);
    }
}

template <typename T, int D, int NT>
void launch(const MQArgs& a, int tiles, int batch, cudaStream_t st) {
    dim3 grid(tiles, a.hkv, batch);
    multi_query_kernel<T, D, NT><<<grid, NW * 32, 0, st>>>(a);
}

// K / V fragments of one block for the pipelined loop (the loads of attend).
template <int D>
struct KVFrag {
    uint4 kr0[D / 32], kr1[D / 32], vr[4][D / 64];
};

template <typename T, int D>
__device__ __forceinline__ void load_k(const T* kb, KVFrag<D>& f, int g, int c) {
#pragma unroll
    for (int i = 0; i < D / 32; ++i) {
        f.kr0[i] = ldg_stream(kb + g * D + 32 * i + 8 * c);
        f.kr1[i] = ldg_stream(kb + (g + 8) * D + 32 * i + 8 * c);
    }
}

template <typename T, int D>
__device__ __forceinline__ void load_v(const T* vb, KVFrag<D>& f, int g, int c) {
#pragma unroll
    for (int j = 0; j < D / 64; ++j) {
        f.vr[0][j] = ldg_stream(vb + (2 * c) * D + 64 * j + 8 * g);
        f.vr[1][j] = ldg_stream(vb + (2 * c + 1) * D + 64 * j + 8 * g);
        f.vr[2][j] = ldg_stream(vb + (8 + 2 * c) * D + 64 * j + 8 * g);
        f.vr[3][j] = ldg_stream(vb + (9 + 2 * c) * D + 64 * j + 8 * g);
    }
}

// attend() for the balanced loop, software-pipelined without extra
// registers: f holds this block's K and V; the next block's K (next_kb) is
// loaded into f as soon as every n-tile's QK^T is done, and its V (next_vb)
// as soon as PV is done, so a block's loads overlap the previous block's
// softmax and PV.  next_kb / next_vb null: nothing to fetch.
template <typename T, int D, int NT>
__device__ __forceinline__ void attend_pipelined(const MQArgs& a, int lb, int ctx, uint32_t qs, const int (&pos)[NT][2],
                                                 MQState<D / 16, NT>& w, KVFrag<D>& f, const T* next_kb,
                                                 const T* next_vb, int g, int c) {
    using H = Half16<T>;
    constexpr int KC = D / 32;
    constexpr int VC = D / 64;
    constexpr int MT = D / 16;
    const int tok0 = lb * BS + g, tok1 = tok0 + 8;
    // ---- S^T = K Q^T for every n-tile, then K is free
    float s[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
        for (int i = 0; i < KC; ++i) {
            const uint4 qf = lds128(qs + (nt * KC + i) * 512);
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                H::mma(s[nt], word(f.kr0[i], 2 * e), word(f.kr1[i], 2 * e), word(f.kr0[i], 2 * e + 1),
                       word(f.kr1[i], 2 * e + 1), word(qf, 2 * e), word(qf, 2 * e + 1));
            }
        }
    }
    if (next_kb) load_k<T, D>(next_kb, f, g, c);

    uint32_t pb0[NT], pb1[NT], pr0[NT], pr1[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const float x0 = tok0 <= pos[nt][0] ? s[nt][0] * a.scale_log2 : neg_inf();
        const float x1 = tok0 <= pos[nt][1] ? s[nt][1] * a.scale_log2 : neg_inf();
        const float x2 = tok1 <= pos[nt][0] ? s[nt][2] * a.scale_log2 : neg_inf();
        const float x3 = tok1 <= pos[nt][1] ? s[nt][3] * a.scale_log2 : neg_inf();
        const float bx0 = fmaxf(x0, x2), bx1 = fmaxf(x1, x3);
        if (__any_sync(0xffffffffu, bx0 > w.m[nt][0] + kSlack || bx1 > w.m[nt][1] + kSlack)) {
            float bm0 = bx0, bm1 = bx1;
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                bm0 = fmaxf(bm0, __shfl_xor_sync(0xffffffffu, bm0, off));
                bm1 = fmaxf(bm1, __shfl_xor_sync(0xffffffffu, bm1, off));
            }
            const float mn0 = fmaxf(w.m[nt][0], bm0), mn1 = fmaxf(w.m[nt][1], bm1);
            const float al0 = mn0 == neg_inf() ? 1.f : ex2(w.m[nt][0] - mn0);
            const float al1 = mn1 == neg_inf() ? 1.f : ex2(w.m[nt][1] - mn1);
            w.l[nt][0] *= al0;
            w.l[nt][1] *= al1;
            w.m[nt][0] = mn0;
            w.m[nt][1] = mn1;
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                w.o[mt][nt][0] *= al0;
                w.o[mt][nt][1] *= al1;
                w.o[mt][nt][2] *= al0;
                w.o[mt][nt][3] *= al1;
            }
        }
        const float r0 = w.m[nt][0] == neg_inf() ? 0.f : w.m[nt][0];
        const float r1 = w.m[nt][1] == neg_inf() ? 0.f : w.m[nt][1];
        const float p0 = ex2(x0 - r0), p1 = ex2(x1 - r1);
        const float p2 = ex2(x2 - r0), p3 = ex2(x3 - r1);
        w.l[nt][0] += p0 + p2;
        w.l[nt][1] += p1 + p3;
        const uint32_t h01 = H::pack(p0, p1), h23 = H::pack(p2, p3);
        pb0[nt] = movmatrix_trans(h01);
        pb1[nt] = movmatrix_trans(h23);
        if constexpr (kSplitP<T>) {
            pr0[nt] = movmatrix_trans(H::pack(p0 - lo_float(h01), p1 - hi_float(h01)));
            pr1[nt] = movmatrix_trans(H::pack(p2 - lo_float(h23), p3 - hi_float(h23)));
        }
    }

    if (lb * BS + BS > ctx) {  // slots past the context may hold any bits
        const int t0 = lb * BS;
#pragma unroll
        for (int j = 0; j < VC; ++j) {
            if (t0 + 2 * c >= ctx) f.vr[0][j] = make_uint4(0, 0, 0, 0);
            if (t0 + 2 * c + 1 >= ctx) f.vr[1][j] = make_uint4(0, 0, 0, 0);
            if (t0 + 8 + 2 * c >= ctx) f.vr[2][j] = make_uint4(0, 0, 0, 0);
            if (t0 + 9 + 2 * c >= ctx) f.vr[3][j] = make_uint4(0, 0, 0, 0);
        }
    }
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
        constexpr int HALF = D / 16;
        const int elo = mt, ehi = mt + HALF;
        const int jl = elo >> 3, wl = (elo & 7) >> 1, hl = elo & 1;
        const int jh = ehi >> 3, wh = (ehi & 7) >> 1, hh = ehi & 1;
        const uint32_t sl = hl ? 0x7632u : 0x5410u;
        const uint32_t sh = hh ? 0x7632u : 0x5410u;
        const uint32_t a0 = __byte_perm(word(f.vr[0][jl], wl), word(f.vr[1][jl], wl), sl);
        const uint32_t a1 = __byte_perm(word(f.vr[0][jh], wh), word(f.vr[1][jh], wh), sh);
        const uint32_t a2 = __byte_perm(word(f.vr[2][jl], wl), word(f.vr[3][jl], wl), sl);
        const uint32_t a3 = __byte_perm(word(f.vr[2][jh], wh), word(f.vr[3][jh], wh), sh);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            H::mma(w.o[mt][nt], a0, a1, a2, a3, pb0[nt], pb1[nt]);
            if constexpr (kSplitP<T>) H::mma(w.o[mt][nt], a0, a1, a2, a3, pr0[nt], pr1[nt]);
        }
    }
    if (next_vb) load_v<T, D>(next_vb, f, g, c);
}

// ------------------------------------------------------------ balanced split
// Calls with at most 24 (query token, query head) rows per (sequence, KV
// head) -- speculative verify of gamma + 1 <= 6 tokens at a GQA group of 4,
// say -- and a workspace take the balanced split of the decode kernels
// (balanced.cuh): warp i streams an equal share of the call's (sequence, KV
// head, 16-token block) items, each warp holding ALL rows of its runs (NT
// n-tiles of 8), so every K/V byte is read once and no warp waits on
// another.  A warp writes one fp32 partial (m, l, o) per row per run it
// touches, at partial row slot * 8 NT + r, slot = i + b * Hkv + kvh; a merge
// kernel behind it (programmatic dependent launch) folds them.
constexpr int kMQWarps = 2;  // warps per CTA of the balanced kernel
constexpr int kMQMaxNT = 3;  // n-tiles of 8 rows per warp, at most
// resident CTAs per SM: as many as the registers of NT n-tiles allow
// (246 / ~190 / 142 registers at D = 128 for NT = 3 / 2 / 1)
constexpr int mq_ctas(int nt) { return nt == 1 ? 6 : 4; }
template <int NT>
constexpr int kMQCtas = mq_ctas(NT);

template <typename T, int D, int NT>
__global__ void __launch_bounds__(kMQWarps * 32, kMQCtas<NT>)
    multi_query_balanced_kernel(MQArgs a, int batch, int nwt_launch, float* ws_o, float* ws_ml) {
    constexpr int KC = D / 32;
    constexpr int MT = D / 16;
    constexpr int R = 8 * NT;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, c = lane & 3;
    // launched behind the previous grid of the stream with programmatic
    // serialization: nothing is read before that grid has completed
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // the merge grid may be scheduled now; it waits for this grid to finish
    asm volatile("griddepcontrol.launch_dependents;");
    // per warp: the run's query fragments ([NT][KC][32] uint4) while it
    // attends, then its R x D partial outputs
    static_assert(R * D >= NT * KC * 32 * 4, "slice too small for the query fragments");
    __shared__ __align__(16) float slice[kMQWarps][R * D];
    uint4* sq = reinterpret_cast<uint4*>(&slice[warp][0]);

    const int i = blockIdx.x * kMQWarps + warp;
    const int cap = a.max_blocks * BS;
    WarpSplit sp;
    bool bad = false;
    const bool any = sp.begin(a.ctx_lens, batch, cap, a.hkv, nwt_launch, kBalancedMinItems, i, bad);
    if (i == 0 && bad && lane == 0) atomicOr(a.status, PKV_STATUS_BAD_CONTEXT);
    if (!any) return;
    while (sp.next()) {
        const int b = sp.b, kvh = sp.kvh, ctx = sp.ctx;
        const int q0 = a.q_start[b], L = a.q_start[b + 1] - q0;
        int rows = L > 0 ? L * a.G : 0;
        if (rows > R || ctx < L) {  // more queries than max_q_len, or fewer tokens than queries
            if (lane == 0 && sp.lb0 == 0) atomicOr(a.status, PKV_STATUS_BAD_CONTEXT);
            rows = rows > R ? R : rows;
        }
        if (rows == 0) continue;
        const int first_pos = ctx - L;

        // query fragments: n-tile nt, column g (row 8 nt + g), k-chunk i
        __syncwarp();  // the previous run's partial rows have been copied out
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int row = 8 * nt + g;
            const T* qrow = nullptr;
            if (row < rows) {
                const int tok = row / a.G, h = row - tok * a.G;
                qrow = static_cast<const T*>(a.q) + ((static_cast<int64_t>(q0) + tok) * a.hq + kvh * a.G + h) * D;
            }
#pragma unroll
            for (int k = 0; k < KC; ++k)
                sq[(nt * KC + k) * 32 + lane] =
                    qrow ? *reinterpret_cast<const uint4*>(qrow + 32 * k + 8 * c) : make_uint4(0, 0, 0, 0);
        }
        __syncwarp();
        const uint32_t qs = static_cast<uint32_t>(__cvta_generic_to_shared(&sq[lane]));
        int pos[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int row = 8 * nt + 2 * c + k;
                const int p = row < rows ? first_pos + row / a.G : -1;
                pos[nt][k] = p < 0 ? -1 : p;
            }
        }

        MQState<MT, NT> w;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            w.m[nt][0] = w.m[nt][1] = neg_inf();
            w.l[nt][0] = w.l[nt][1] = 0.f;
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
                w.o[mt][nt][0] = w.o[mt][nt][1] = w.o[mt][nt][2] = w.o[mt][nt][3] = 0.f;
        }
        const int32_t* trow = a.tables + static_cast<int64_t>(b) * a.max_blocks;
        // Block k of the run has id shfl(tab, k % 32); lane j of tab holds
        // the id of the run's block 32 (k / 32) + j.  One block ahead: block
        // k + 1's K and V are fetched while block k is attended.
        const T* kpool = static_cast<const T*>(a.k_pool);
        const T* vpool = static_cast<const T*>(a.v_pool);
        auto base_of = [&](int phys) { return (static_cast<int64_t>(phys) * a.hkv + kvh) * (BS * D); };
        auto valid = [&](int phys) { return static_cast<unsigned>(phys) < static_cast<unsigned>(a.num_blocks); };
        int tab = sp.lb0 + lane < sp.lb1 ? trow[sp.lb0 + lane] : -1;
        int phys = __shfl_sync(0xffffffffu, tab, 0);
        KVFrag<D> f;
        if (valid(phys)) {
            load_k<T, D>(kpool + base_of(phys), f, g, c);
            load_v<T, D>(vpool + base_of(phys), f, g, c);
        }
        for (int lb = sp.lb0, k = 0; lb < sp.lb1; ++lb, ++k) {
            int pn = -1;
            if (lb + 1 < sp.lb1) {
                if (((k + 1) & 31) == 0) {  // ids of the run's next 32 blocks
                    const int idx = lb + 1 + lane;
                    tab = idx < sp.lb1 ? trow[idx] : -1;
                }
                pn = __shfl_sync(0xffffffffu, tab, (k + 1) & 31);
            }
            const bool nv = valid(pn);
            if (!valid(phys)) {
                if (lane == 0) atomicOr(a.status, PKV_STATUS_BAD_BLOCK);
                if (nv) {  // nothing attended: fetch the next block now
                    load_k<T, D>(kpool + base_of(pn), f, g, c);
                    load_v<T, D>(vpool + base_of(pn), f, g, c);
                }
            } else {
                attend_pipelined<T, D, NT>(a, lb, ctx, qs, pos, w, f, nv ? kpool + base_of(pn) : nullptr,
                                           nv ? vpool + base_of(pn) : nullptr, g, c);
            }
            phys = pn;
        }

        // ---- the run's partial rows: l totalled over the token lanes, o
        // staged through the slice so rows go out in 16-byte stores
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                w.l[nt][0] += __shfl_xor_sync(0xffffffffu, w.l[nt][0], off);
                w.l[nt][1] += __shfl_xor_sync(0xffffffffu, w.l[nt][1], off);
            }
        }
        __syncwarp();  // the query fragments are no longer read
        float* so = &slice[warp][0];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            const int dl = pv_col(mt, g), dh = pv_col(mt + D / 16, g);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                so[(8 * nt + 2 * c) * D + dl] = w.o[mt][nt][0];
                so[(8 * nt + 2 * c + 1) * D + dl] = w.o[mt][nt][1];
                so[(8 * nt + 2 * c) * D + dh] = w.o[mt][nt][2];
                so[(8 * nt + 2 * c + 1) * D + dh] = w.o[mt][nt][3];
            }
        }
        __syncwarp();
        const int64_t slot = i + static_cast<int64_t>(b) * a.hkv + kvh;
        float4* po = reinterpret_cast<float4*>(ws_o + slot * R * D);
        const float4* s4 = reinterpret_cast<const float4*>(so);
        for (int x = lane; x < rows * D / 4; x += 32) po[x] = s4[x];
        if (g == 0) {
            float* pml = ws_ml + slot * R * 2;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const int row = 8 * nt + 2 * c + k;
                    if (row < rows) {
                        pml[2 * row] = w.m[nt][k];
                        pml[2 * row + 1] = w.l[nt][k];
                    }
                }
            }
        }
    }
}

// Merge of a balanced multi-query split: one CTA of kMergeThreads threads
// per (sequence, KV head) folds the partials of all its rows: for each (row,
// column), the partials of the consecutive warps whose ranges met the run,
// with a log-sum-exp rescale.  Where the run sits among the items follows
// from the context lengths alone (inputs of the call), so it is worked out
// before the wait on the split grid.
constexpr int kMergeThreads = 256;

template <typename T, int D, int NT>
__global__ void __launch_bounds__(kMergeThreads) multi_query_merge_kernel(
    const int32_t* __restrict__ q_start, const int32_t* __restrict__ ctx_lens, int batch, int hq, int hkv,
    int cap, int nwt_launch, const float* __restrict__ ws_o, const float* __restrict__ ws_ml, T* __restrict__ out) {
    constexpr int R = 8 * NT, NWARP = kMergeThreads / 32;
    const int kvh = blockIdx.x, b = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int G = hq / hkv;
    int before = 0, total = 0;
    for (int j = tid; j < batch; j += kMergeThreads) {
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
    const int q0 = q_start[b], L = q_start[b + 1] - q0;
    const int rows = L > 0 ? (L * G < R ? L * G : R) : 0;
    if (rows == 0) return;
    const int nb = blocks_of(ctx_lens[b], cap);
    const int W = total * hkv;
    const int nwt = max(min(W / kBalancedMinItems, nwt_launch), 1);
    const int S = before * hkv + kvh * nb;
    int64_t slot0 = 0;
    int np = 0;
    if (nb > 0) {
        const int64_t i0 = first_warp(S, W, nwt), i1 = first_warp(S + nb - 1, W, nwt);
        slot0 = i0 + static_cast<int64_t>(b) * hkv + kvh;
        np = static_cast<int>(i1 - i0 + 1);
    }
    // partials are produced by the preceding grid: wait for it
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // 1. per row: M = max_p m_p and 1 / L, L = sum_p l_p 2^(m_p - M) (one
    // warp per row, lanes over the partials)
    __shared__ float rowM[R], rowInv[R];
    const float* ml = ws_ml + slot0 * R * 2;  // partial p, row r: ml[(p R + r) 2 + {0, 1}]
    for (int r = warp; r < rows; r += NWARP) {
        float M = neg_inf();
        for (int p = lane; p < np; p += 32) M = fmaxf(M, __ldcg(ml + (static_cast<int64_t>(p) * R + r) * 2));
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
        float L = 0.f;
        if (M != neg_inf()) {
            for (int p = lane; p < np; p += 32) {
                const float* e = ml + (static_cast<int64_t>(p) * R + r) * 2;
                L += __ldcg(e + 1) * ex2(__ldcg(e) - M);
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
        if (lane == 0) {
            rowM[r] = M;
            rowInv[r] = L > 0.f ? 1.f / L : 0.f;
        }
    }
    __syncthreads();
    // 2. out[r, d..d+3] = sum_p 2^(m_p - M) o_p[r, d..d+3] / L: 16-byte
    // partial loads (the threads of a row share each m_p load)
    constexpr int D4 = D / 4;
    for (int x = tid; x < rows * D4; x += kMergeThreads) {
        const int r = x / D4, d = (x - r * D4) * 4;
        const int tok = r / G, h = r - tok * G;
        const float M = rowM[r], inv = rowInv[r];
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (inv > 0.f) {
            for (int p = 0; p < np; ++p) {
                const int64_t row = (slot0 + p) * R + r;
                const float w = ex2(__ldcg(ws_ml + row * 2) - M);
                const float4 o = __ldcg(reinterpret_cast<const float4*>(ws_o + row * D + d));
                acc.x += w * o.x;
                acc.y += w * o.y;
                acc.z += w * o.z;
                acc.w += w * o.w;
            }
        }
        uint2 v;
        v.x = Half16<T>::pack(acc.x * inv, acc.y * inv);
        v.y = Half16<T>::pack(acc.z * inv, acc.w * inv);
        *reinterpret_cast<uint2*>(out + ((static_cast<int64_t>(q0) + tok) * hq + kvh * G + h) * D + d) = v;
    }
}

// Warps the balanced multi-query split launches for NT n-tiles.
int mq_warps(int64_t max_items, int nt) {
    return balanced_warps(max_items, kMQWarps * mq_ctas(nt));
}

// n-tiles of the balanced split for rows per (sequence, KV head), 0 if it
// does not apply (more than 24 rows, more than 1,024 sequences, or too few
// items per launched warp).
int mq_balanced_nt(int64_t batch, int64_t hkv, int64_t max_blocks, int64_t rows) {
    if (rows <= 0 || rows > 8 * kMQMaxNT || batch > kBalancedMaxBatch) return 0;
    const int nt = static_cast<int>((rows + 7) / 8);
    const int64_t items = batch * hkv * max_blocks;
    if (items >= (1LL << 30)) return 0;
    const int per_sm = kMQWarps * mq_ctas(nt);
    if (items < static_cast<int64_t>(kBalancedItemsPerWarp) * per_sm * num_sms()) return 0;
    return nt;
}

size_t mq_balanced_bytes(int64_t batch, int64_t hkv, int D, int nt, int nwt) {
    return static_cast<size_t>(nwt + batch * hkv) * 8 * nt * (D + 2) * sizeof(float);
}

template <typename T, int D, int NT>
int run_mq_balanced(const MQArgs& a, int batch, int nwt, float* ws_o, float* ws_ml, cudaStream_t st) {
    {
        cudaLaunchConfig_t c0 = {};
        c0.gridDim = dim3((nwt + kMQWarps - 1) / kMQWarps);
        c0.blockDim = dim3(kMQWarps * 32);
        c0.stream = st;
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        at[0].val.programmaticStreamSerializationAllowed = 1;
        c0.attrs = at;
        c0.numAttrs = 1;
        if (cudaLaunchKernelEx(&c0, multi_query_balanced_kernel<T, D, NT>, a, batch, nwt, ws_o, ws_ml) != cudaSuccess)
            return PKV_ERR_CUDA;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.hkv, batch);
    cfg.blockDim = dim3(kMergeThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, multi_query_merge_kernel<T, D, NT>, a.q_start, a.ctx_lens, batch,
                                             a.hq, a.hkv, a.max_blocks * BS, nwt,
                                             static_cast<const float*>(ws_o), static_cast<const float*>(ws_ml),
                                             static_cast<T*>(a.out));
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

template <typename T, int D>
int dispatch_mq_balanced(const MQArgs& a, int batch, int nt, int nwt, float* ws_o, float* ws_ml, cudaStream_t st) {
    if (nt == 1) return run_mq_balanced<T, D, 1>(a, batch, nwt, ws_o, ws_ml, st);
    if (nt == 2) return run_mq_balanced<T, D, 2>(a, batch, nwt, ws_o, ws_ml, st);
    return run_mq_balanced<T, D, 3>(a, batch, nwt, ws_o, ws_ml, st);
}

template <typename T, int D>
void launch_nt(const MQArgs& a, int rows, int batch, cudaStream_t st) {
    if (rows <= 8) launch<T, D, 1>(a, 1, batch, st);
    else launch<T, D, 2>(a, (rows + 15) / 16, batch, st);
}

}  // namespace
}  // namespace pkv

extern "C" int pkv_multi_query_workspace_bytes(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                               int32_t head_dim, int32_t max_blocks, int32_t block_size,
                                               int32_t max_q_len, size_t* out) {
    if (!out || batch < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || max_blocks < 0 ||
        block_size <= 0 || max_q_len < 0 || num_q_heads % num_kv_heads != 0)
        return PKV_ERR_INVALID_ARG;
    if (block_size != pkv::BS) return PKV_ERR_UNSUPPORTED;
    const int64_t rows = static_cast<int64_t>(max_q_len) * (num_q_heads / num_kv_heads);
    const int nt = pkv::mq_balanced_nt(batch, num_kv_heads, max_blocks, rows);
    if (nt == 0) {
        *out = 0;
        return PKV_OK;
    }
    const int nwt = pkv::mq_warps(static_cast<int64_t>(batch) * num_kv_heads * max_blocks, nt);
    *out = pkv::mq_balanced_bytes(batch, num_kv_heads, head_dim, nt, nwt);
    return PKV_OK;
}

extern "C" int pkv_paged_attention_multi_query(
    const void* q, const int32_t* q_start, const void* k_pool, const void* v_pool,
    const int32_t* block_tables, const int32_t* context_lens, int32_t batch, int32_t num_q_heads,
    int32_t num_kv_heads, int32_t head_dim, int32_t num_blocks, int32_t block_size,
    int32_t max_blocks, int32_t max_q_len, float scale, void* out, void* workspace,
    size_t workspace_bytes, int dtype, void* stream) {
    if (batch < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || num_blocks <= 0 ||
        block_size <= 0 || max_blocks < 0 || max_q_len < 0)
        return PKV_ERR_INVALID_ARG;
    if (dtype != PKV_DTYPE_F16 && dtype != PKV_DTYPE_BF16) return PKV_ERR_INVALID_ARG;
    if (num_q_heads % num_kv_heads != 0) return PKV_ERR_INVALID_ARG;
    if (block_size != pkv::BS || (head_dim != 64 && head_dim != 128) || num_q_heads / num_kv_heads > 8 ||
        batch > 65535 || num_kv_heads > 65535)
        return PKV_ERR_UNSUPPORTED;
    const int64_t rows = static_cast<int64_t>(max_q_len) * (num_q_heads / num_kv_heads);
    if (rows > 16LL * 65535) return PKV_ERR_UNSUPPORTED;
    if (batch == 0 || max_q_len == 0) return PKV_OK;
    if (!q || !q_start || !k_pool || !v_pool || !block_tables || !context_lens || !out)
        return PKV_ERR_INVALID_ARG;
    if (!pkv::aligned16(q) || !pkv::aligned16(k_pool) || !pkv::aligned16(v_pool) || !pkv::aligned16(out) ||
        (reinterpret_cast<uintptr_t>(q_start) & 3u) || (reinterpret_cast<uintptr_t>(block_tables) & 3u) ||
        (reinterpret_cast<uintptr_t>(context_lens) & 3u))
        return PKV_ERR_MISALIGNED;
    int* st = pkv::status_word();
    if (!st) return PKV_ERR_CUDA;
    pkv::MQArgs a;
    a.q = q;
    a.q_start = q_start;
    a.k_pool = k_pool;
    a.v_pool = v_pool;
    a.tables = block_tables;
    a.ctx_lens = context_lens;
    a.hq = num_q_heads;
    a.hkv = num_kv_heads;
    a.G = num_q_heads / num_kv_heads;
    a.num_blocks = num_blocks;
    a.max_blocks = max_blocks;
    a.scale_log2 = scale * pkv::kLog2e;
    a.out = out;
    a.status = st;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    const int r = static_cast<int>(rows);
    // with a workspace, the balanced split where it applies
    const int nt = workspace ? pkv::mq_balanced_nt(batch, num_kv_heads, max_blocks, rows) : 0;
    if (nt > 0) {
        const int nwt = pkv::mq_warps(static_cast<int64_t>(batch) * num_kv_heads * max_blocks, nt);
        if (workspace_bytes < pkv::mq_balanced_bytes(batch, num_kv_heads, head_dim, nt, nwt))
            return PKV_ERR_WORKSPACE;
        if (!pkv::aligned16(workspace)) return PKV_ERR_MISALIGNED;
        float* ws_o = static_cast<float*>(workspace);
        float* ws_ml = ws_o + static_cast<size_t>(nwt + static_cast<int64_t>(batch) * num_kv_heads) * 8 * nt *
                                  head_dim;
        if (dtype == PKV_DTYPE_BF16) {
            return head_dim == 128 ? pkv::dispatch_mq_balanced<__nv_bfloat16, 128>(a, batch, nt, nwt, ws_o, ws_ml, cs)
                                   : pkv::dispatch_mq_balanced<__nv_bfloat16, 64>(a, batch, nt, nwt, ws_o, ws_ml, cs);
        }
        return head_dim == 128 ? pkv::dispatch_mq_balanced<__half, 128>(a, batch, nt, nwt, ws_o, ws_ml, cs)
                               : pkv::dispatch_mq_balanced<__half, 64>(a, batch, nt, nwt, ws_o, ws_ml, cs);
    }
    // long query spans (chunked-prefill slices): the tensor-core kernel
    if (pkv::prefill_tc_applies(head_dim, num_q_heads / num_kv_heads, rows))
        return pkv::launch_prefill_tc(q, q_start, k_pool, v_pool, block_tables, context_lens, batch, num_q_heads,
                                      num_kv_heads, num_blocks, max_blocks, max_q_len, scale, out, st,
                                      dtype == PKV_DTYPE_BF16, cs);
    if (dtype == PKV_DTYPE_BF16) {
        if (head_dim == 128) pkv::launch_nt<__nv_bfloat16, 128>(a, r, batch, cs);
        else pkv::launch_nt<__nv_bfloat16, 64>(a, r, batch, cs);
    } else {
        if (head_dim == 128) pkv::launch_nt<__half, 128>(a, r, batch, cs);
        else pkv::launch_nt<__half, 64>(a, r, batch, cs);
    }
    return pkv::launch_status();
}
