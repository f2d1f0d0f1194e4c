// Paged decode attention over an INT4-asymmetric or FP8-E4M3 KV cache with
// 16-bit attention sinks.
//
// What it computes: the decode attention of decode.cu with every cached
// K/V value replaced by its dequantised value -- (q - z) * s for INT4, with
// one fp16 (s, z) per (token, head) (group = head dim); e4m3(code) * s for
// FP8, one fp16 s per (token, head) -- except the first n_sink positions of
// each sequence, which read the 16-bit sink buffers ("The 8GB VRAM
// Breakthrough", §4 "The Hybrid Solution: Sink-FP16 + Group-Wise Asymmetric
// INT4 / FP8"; §5 "On-the-Fly Register Dequantization": packed codes and
// (scale, zero) go straight to registers, no dequantised copy in memory).
//
// Design: the tensor-core layout of decode.cu (tokens as M for QK^T, head dim
// as M for PV, the GQA group as N), with fragments built from the codes in
// registers and the per-token scale / zero factored out of the products:
//   QK^T: S_t = s_t * (sum_d q_d c_td - z_t * sum_d q_d)   INT4
//         S_t = s_t * sum_d q_d e4m3(c_td)                 FP8
//   PV:   O_d = sum_t W_t c_td - sum_t W_t z_t,  W_t = P_t s_t
// so the MMAs see exact code values against fp16 queries / weights, with
// fp32 accumulation.
//   INT4 codes -> fp16 with one AND per pair: a nibble c in the low bits of
//   a 16-bit half is the fp16 subnormal c x 2^-24 (exact), the next nibble up
//   is 16 c x 2^-24.  A 32-bit word of 8 nibbles yields four pairs
//   {d_j, d_j+4}: masks 0x000F000F / 0x00F000F0 on the word and on the word
//   shifted by 8.  The k order of a k-step is permuted accordingly; the
//   query columns that meet the 16x nibbles go in divided by 16, and the PV
//   accumulator columns fed by them are scaled back by 2^20 (the others by
//   2^24) at the end.
//   FP8 -> fp16: cvt.rn.f16x2.e4m3x2 (exact).
//   For PV the pairs must hold two tokens of one column: a byte permute of
//   the two token rows' words comes first.
// Online softmax: the warp-wide block max is exact; the rescale of o, l and
// the zero-point correction is skipped when no max changed (the usual case
// once a few blocks are in).
// Sink tokens (positions < n_sink <= 16, i.e. in logical block 0): their
// logits are recomputed in fp32 from the 16-bit sink keys, their PV weights
// are zero in the MMA, and P * sink_v is added to the accumulator directly.

#include <type_traits>

#include "balanced.cuh"

namespace pkv {
namespace {

constexpr int BS = 16;
constexpr int NW = 4;
// INT4 runs 5 CTAs per SM (96 registers) with the query fragments re-read
// from shared memory per block (4 with two column groups, whose per-group
// sums, scales and weights need the registers); FP8 needs its registers for
// the 4 KiB of codes per block and keeps 4 CTAs with the query fragments in
// registers.
// (Measured on the 32 x 16k workload: INT4 259 -> 242 us; FP8 unchanged or
// slower with the INT4 settings.)
template <int QMODE, int NG = 1, bool PAIR = false>
constexpr int kCtasPerSm = PAIR ? 4 : (QMODE == PKV_QMODE_INT4_ASYM && NG == 1 ? 5 : 4);
template <int QMODE>
constexpr bool kQueryInShared = QMODE == PKV_QMODE_INT4_ASYM;
constexpr float kLog2e = 1.4426950408889634f;
// Headroom (log2 units) a logit may rise above the running reference max
// before the online softmax rescales: weights stay <= 2^8 (fp16-safe).
constexpr float kSlack = 8.f;
// Largest V scale for which a weight of 2^kSlack keeps W = P s well inside
// fp16 (65,504): blocks with a larger one take the exact max.
constexpr float kLazyMaxScale = 128.f;

struct QDecodeArgs {
    const void* q;
    const uint8_t* k_codes;
    const __half* k_scale;
    const __half* k_zero;
    const uint8_t* v_codes;
    const __half* v_scale;
    const __half* v_zero;
    const void* sink_k;
    const void* sink_v;
    int n_sink;
    const void* win_k;   // 16-bit window rings [rows, ring, Hkv, 16, D] (window > 0)
    const void* win_v;
    int window, ring;
    const int32_t* tables;
    const int32_t* ctx_lens;
    int hq, hkv, G, num_blocks, max_blocks, part_blocks, max_parts;
    float scale_log2;
    void* out;
    float* ws_o;
    float* ws_ml;
    int* status;
};

__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
    Half16<__half>::mma(d, a0, a1, a2, a3, b0, b1);
}

__device__ __forceinline__ uint32_t f16pair(float lo, float hi) { return Half16<__half>::pack(lo, hi); }

// INT4 nibbles as fp16 subnormals: masking a 32-bit word with 0x000F000F
// leaves the nibbles at bits 0 and 16 as the fp16 pair {n_lo, n_hi} x 2^-24,
// exactly; the mask 0x00F000F0 leaves the next nibbles as {16 n_lo, 16 n_hi}
// x 2^-24.  One logic op per pair, no float arithmetic: the 2^-24 (and the 16
// of the odd nibbles) are taken out after the products.
__device__ __forceinline__ uint32_t nib_even(uint32_t w) { return w & 0x000F000Fu; }
__device__ __forceinline__ uint32_t nib_odd(uint32_t w) { return w & 0x00F000F0u; }
constexpr float kTwo24 = 16777216.f;         // 2^24
constexpr float kInvTwo24 = 5.9604645e-08f;  // 2^-24

// 16-byte shared load, kept in place (not hoisted out of the block loop).
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 r;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "r"(addr));
    return r;
}

// two e4m3 codes in the low 16 bits of w -> fp16 pair (low byte -> low half)
__device__ __forceinline__ uint32_t e4m3x2(uint32_t w) {
    uint32_t d;
    const unsigned short a = static_cast<unsigned short>(w & 0xffffu);
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(d) : "h"(a));
    return d;
}

template <typename T>
__device__ __forceinline__ float tofloat(T x) {
    return Half16<T>::to_float(x);
}

// Online-softmax state of one warp over the blocks it attended, for the
// query heads 2c, 2c+1 of its lanes: per-lane partial sums l and (INT4) the
// zero-point correction sum_t W_t z_t, and the PV accumulator in the MMA's
// units (INT4: 2^-24, odd columns 2^-20).
template <int MT, int NG>
struct QState {
    float m0, m1, l0, l1;
    float corr[NG][2];  // per column group, heads 2c / 2c + 1
    float o[MT][4];
    bool true_units;    // o already in true units (a window block was attended)
    __device__ __forceinline__ void init() {
        m0 = m1 = neg_inf();
        l0 = l1 = 0.f;
        true_units = false;
#pragma unroll
        for (int gi = 0; gi < NG; ++gi) corr[gi][0] = corr[gi][1] = 0.f;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
    }
};

// PV element e (0 .. D/8 - 1) of m-tile mt, half hf (M rows g / g + 8).  One
// column group (NG = 1): e = mt, mt + MT.  Two groups of 64 columns (NG = 2):
// e = 8 (mt / 4) + mt % 4 + 4 hf, so both halves of an m-tile lie in one
// group and take that group's weights.  Both halves have the same parity.
template <int NG, int MT>
__host__ __device__ constexpr int pv_e(int mt, int hf) {
    return NG == 1 ? mt + hf * MT : 8 * (mt / 4) + mt % 4 + 4 * hf;
}
// Head-dim column of element e of lane group g: NG = 1, the lane's DS
// consecutive columns; NG = 2, 8 columns in each 64-column group.
template <int NG, int D>
__device__ __forceinline__ int pv_column(int e, int g) {
    return NG == 1 ? g * (D / 8) + e : (e >> 3) * 64 + 8 * g + (e & 7);
}

// The quantised blocks of a pass two at a time (INT4, G <= 4; the scheme is
// described at quant_pass), the two column halves merged, then the window
// blocks one by one with attend16.  qs: the shared query slices (two
// copies); qs0, qs1: the group sums of the lane's query heads 2 hh, 2 hh + 1.
template <typename T, int D, int NG, bool WIN, typename Attend16>
__device__ __forceinline__ void quant_pairs(const QDecodeArgs& a, int b, int kvh, int ctx, int lb_first,
                                            int lb_end, int stride, int win_lb0, uint32_t qs,
                                            const float (&qs0)[NG], const float (&qs1)[NG],
                                            QState<D / 16, NG>& st, Attend16& attend16) {
    constexpr int KSTEPS = D / 16;
    constexpr int MT = D / 16;
    constexpr int CB = D / 2;        // code bytes per row
    constexpr int KW = D / 32;       // 32-bit K-code words per lane per row
    constexpr int VW = D / 64;       // 32-bit V-code words per lane per row
    constexpr int DS = D / 8;
    constexpr int KPG = KW / NG;
    constexpr int VPG = VW / NG;
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
    const int sl = c >> 1;           // the lane's column half: block A (0) or B (1)
    const int hh = c & 1;
    float& m0 = st.m0;
    float& m1 = st.m1;
    float& l0 = st.l0;
    float& l1 = st.l1;
    auto& corr = st.corr;
    auto& o = st.o;
    const int32_t* trow = a.tables + static_cast<int64_t>(b) * a.max_blocks;
    const int vr0 = 2 * c, vr1 = 2 * c + 1, vr2 = 8 + 2 * c, vr3 = 9 + 2 * c;

    struct Codes {
        uint32_t kw0[KW], kw1[KW], vw[4][VW];
    };
    struct Scales {
        __half2 ks[NG], vs[NG], kz[NG], vz[NG];  // low: token g, high: token g + 8
    };
    // Per-lane base addresses for this pass's KV head; a block adds
    // phys x (the pool's bytes per block) with one widening multiply-add,
    // and every load of the block is an immediate offset from it.
    const uint32_t code_stride = static_cast<uint32_t>(a.hkv) * (BS * CB);      // bytes per pool block
    const uint32_t scale_stride = static_cast<uint32_t>(a.hkv) * (BS * NG * 2);  // bytes per pool block
    const uint8_t* kbase = a.k_codes + static_cast<uint32_t>(kvh) * (BS * CB) + g * CB +
                           (NG == 2 ? 8 * c : (KW == 4 ? 16 * c : 8 * c));
    const uint8_t* vbase = a.v_codes + static_cast<uint32_t>(kvh) * (BS * CB) + vr0 * CB +
                           (NG == 2 ? 4 * g : DS / 2 * g);
    const uint32_t soff = (static_cast<uint32_t>(kvh) * BS + g) * (NG * 2);  // bytes, token g
    const uint8_t* ksb = reinterpret_cast<const uint8_t*>(a.k_scale) + soff;
    const uint8_t* vsb = reinterpret_cast<const uint8_t*>(a.v_scale) + soff;
    const uint8_t* kzb = reinterpret_cast<const uint8_t*>(a.k_zero) + soff;
    const uint8_t* vzb = reinterpret_cast<const uint8_t*>(a.v_zero) + soff;
    auto at = [](const uint8_t* base, int phys, uint32_t stride) {
        return base + static_cast<uint64_t>(static_cast<uint32_t>(phys)) * stride;
    };
    auto load_codes = [&](int phys, Codes& C) {
        const uint8_t* kc = at(kbase, phys, code_stride);  // row g, this lane's columns
        const uint8_t* vc = at(vbase, phys, code_stride);  // row 2c, this lane's columns
        // V rows 2c + 1, 8 + 2c, 9 + 2c are 1, 8, 9 rows further
        if constexpr (NG == 2) {
#pragma unroll
            for (int gi = 0; gi < 2; ++gi) {
                const uint2 r0 = ldg_stream8(kc + 32 * gi);
                const uint2 r1 = ldg_stream8(kc + 8 * CB + 32 * gi);
                C.kw0[2 * gi] = r0.x; C.kw0[2 * gi + 1] = r0.y;
                C.kw1[2 * gi] = r1.x; C.kw1[2 * gi + 1] = r1.y;
                C.vw[0][gi] = *reinterpret_cast<const uint32_t*>(vc + 32 * gi);
                C.vw[1][gi] = *reinterpret_cast<const uint32_t*>(vc + CB + 32 * gi);
                C.vw[2][gi] = *reinterpret_cast<const uint32_t*>(vc + 8 * CB + 32 * gi);
                C.vw[3][gi] = *reinterpret_cast<const uint32_t*>(vc + 9 * CB + 32 * gi);
            }
        } else {
            if constexpr (KW == 4) {
                const uint4 r0 = ldg_stream(kc);
                const uint4 r1 = ldg_stream(kc + 8 * CB);
                C.kw0[0] = r0.x; C.kw0[1] = r0.y; C.kw0[2] = r0.z; C.kw0[3] = r0.w;
                C.kw1[0] = r1.x; C.kw1[1] = r1.y; C.kw1[2] = r1.z; C.kw1[3] = r1.w;
            } else {
                const uint2 r0 = ldg_stream8(kc);
                const uint2 r1 = ldg_stream8(kc + 8 * CB);
                C.kw0[0] = r0.x; C.kw0[1] = r0.y;
                C.kw1[0] = r1.x; C.kw1[1] = r1.y;
            }
            if constexpr (VW == 2) {
                const uint2 x0 = ldg_stream8(vc), x1 = ldg_stream8(vc + CB);
                const uint2 x2 = ldg_stream8(vc + 8 * CB), x3 = ldg_stream8(vc + 9 * CB);
                C.vw[0][0] = x0.x; C.vw[0][1] = x0.y; C.vw[1][0] = x1.x; C.vw[1][1] = x1.y;
                C.vw[2][0] = x2.x; C.vw[2][1] = x2.y; C.vw[3][0] = x3.x; C.vw[3][1] = x3.y;
            } else {
                C.vw[0][0] = *reinterpret_cast<const uint32_t*>(vc);
                C.vw[1][0] = *reinterpret_cast<const uint32_t*>(vc + CB);
                C.vw[2][0] = *reinterpret_cast<const uint32_t*>(vc + 8 * CB);
                C.vw[3][0] = *reinterpret_cast<const uint32_t*>(vc + 9 * CB);
            }
        }
    };
    // the scales and zero points of the lane's own block (tokens g, g + 8)
    auto load_scales = [&](int phys, Scales& S) {
        const __half* ks = reinterpret_cast<const __half*>(at(ksb, phys, scale_stride));
        const __half* vs = reinterpret_cast<const __half*>(at(vsb, phys, scale_stride));
        const __half* kz = reinterpret_cast<const __half*>(at(kzb, phys, scale_stride));
        const __half* vz = reinterpret_cast<const __half*>(at(vzb, phys, scale_stride));
#pragma unroll
        for (int gi = 0; gi < NG; ++gi) {
            S.ks[gi] = __halves2half2(ks[gi], ks[8 * NG + gi]);
            S.vs[gi] = __halves2half2(vs[gi], vs[8 * NG + gi]);
            S.kz[gi] = __halves2half2(kz[gi], kz[8 * NG + gi]);
            S.vz[gi] = __halves2half2(vz[gi], vz[8 * NG + gi]);
        }
    };
    // PV A fragment of element e (token pair pr) from a block's V words
    auto pv_frag = [&](const Codes& C, int e, int pr) {
        const uint32_t* R0 = C.vw[2 * pr];
        const uint32_t* R1 = C.vw[2 * pr + 1];
        const int word = e >> 3, sub = (e >> 2) & 1, nib = e & 3;
        const uint32_t X = __byte_perm(R0[word], R1[word], sub ? 0x7632u : 0x5410u);
        const uint32_t Y = nib >= 2 ? X >> 8 : X;
        return (nib & 1) ? nib_odd(Y) : nib_even(Y);
    };

    auto attend_pair = [&](int lbA, bool vA, bool vB, const Codes& CA, const Codes& CB, const Scales& S) {
        // ---- S^T = C Q^T: block A against the query in columns 0-3, block B
        // against it in columns 4-7, one accumulator per column group
        float sg[NG][4];
#pragma unroll
        for (int gi = 0; gi < NG; ++gi) sg[gi][0] = sg[gi][1] = sg[gi][2] = sg[gi][3] = 0.f;
#pragma unroll
        for (int k = 0; k < KW; ++k) {
            const uint4 qa = lds128(qs + k * 512);
            const uint4 qb = lds128(qs + (KSTEPS / 2 + k) * 512);
            float (&sk)[4] = sg[k / KPG];
            const uint32_t a0 = CA.kw0[k] >> 8, a1 = CA.kw1[k] >> 8;
            mma_f16(sk, nib_even(CA.kw0[k]), nib_even(CA.kw1[k]), nib_odd(CA.kw0[k]), nib_odd(CA.kw1[k]),
                    qa.x, qa.y);
            mma_f16(sk, nib_even(a0), nib_even(a1), nib_odd(a0), nib_odd(a1), qa.z, qa.w);
            const uint32_t b0 = CB.kw0[k] >> 8, b1 = CB.kw1[k] >> 8;
            mma_f16(sk, nib_even(CB.kw0[k]), nib_even(CB.kw1[k]), nib_odd(CB.kw0[k]), nib_odd(CB.kw1[k]),
                    qb.x, qb.y);
            mma_f16(sk, nib_even(b0), nib_even(b1), nib_odd(b0), nib_odd(b1), qb.z, qb.w);
        }
        // ---- the lane's block: A for c = 0, 1, B for c = 2, 3
        const int lbm = lbA + (sl ? stride : 0);
        const bool vm = sl ? vB : vA;
        const int t0 = lbm * BS;
        const bool ok0 = vm && t0 + g < ctx, ok1 = vm && t0 + g + 8 < ctx;
        float x0 = 0.f, x1 = 0.f, x2 = 0.f, x3 = 0.f;
#pragma unroll
        for (int gi = 0; gi < NG; ++gi) {
            const float ks0 = __low2float(S.ks[gi]), ks1 = __high2float(S.ks[gi]);
            const float kz0 = __low2float(S.kz[gi]), kz1 = __high2float(S.kz[gi]);
            x0 += ks0 * (sg[gi][0] * kTwo24 - kz0 * qs0[gi]);
            x1 += ks0 * (sg[gi][1] * kTwo24 - kz0 * qs1[gi]);
            x2 += ks1 * (sg[gi][2] * kTwo24 - kz1 * qs0[gi]);
            x3 += ks1 * (sg[gi][3] * kTwo24 - kz1 * qs1[gi]);
        }
        x0 *= a.scale_log2;
        x1 *= a.scale_log2;
        x2 *= a.scale_log2;
        x3 *= a.scale_log2;
        // sinks: only logical block 0, which is block A of a pass's first step
        const bool sinks_here = lbA == 0 && a.n_sink > 0;
        bool sk0 = false, sk1 = false;
        if (sinks_here) {
            sk0 = sl == 0 && g < a.n_sink;
            sk1 = sl == 0 && g + 8 < a.n_sink;
            const T* qbase = static_cast<const T*>(a.q) + (static_cast<int64_t>(b) * a.hq + kvh * a.G) * D;
            const T* skb = static_cast<const T*>(a.sink_k);
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int t = g + 8 * r;
                if (sl == 0 && t < a.n_sink) {
                    const T* krow = skb + ((static_cast<int64_t>(b) * a.n_sink + t) * a.hkv + kvh) * D;
                    float d0 = 0.f, d1 = 0.f;
                    const int h0 = min(2 * hh, a.G - 1), h1 = min(2 * hh + 1, a.G - 1);
                    for (int d = 0; d < D; ++d) {
                        const float kv = tofloat(krow[d]);
                        d0 += tofloat(qbase[h0 * D + d]) * kv;
                        d1 += tofloat(qbase[h1 * D + d]) * kv;
                    }
                    if (r == 0) {
                        x0 = d0 * a.scale_log2;
                        x1 = d1 * a.scale_log2;
                    } else {
                        x2 = d0 * a.scale_log2;
                        x3 = d1 * a.scale_log2;
                    }
                }
            }
        }
        if (!ok0) x0 = x1 = neg_inf();
        if (!ok1) x2 = x3 = neg_inf();

        // ---- online softmax of the lane's stream (as in quant_pass)
        const float bx0 = fmaxf(x0, x2), bx1 = fmaxf(x1, x3);
        float vsmax = 0.f;
#pragma unroll
        for (int gi = 0; gi < NG; ++gi)
            vsmax = fmaxf(vsmax, fmaxf(__low2float(S.vs[gi]), __high2float(S.vs[gi])));
        if (__any_sync(0xffffffffu, bx0 > m0 + kSlack || bx1 > m1 + kSlack || vsmax > kLazyMaxScale)) {
            float bm0 = bx0, bm1 = bx1;
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                bm0 = fmaxf(bm0, __shfl_xor_sync(0xffffffffu, bm0, off));
                bm1 = fmaxf(bm1, __shfl_xor_sync(0xffffffffu, bm1, off));
            }
            // a stream may have had no live token yet (its maxima still
            // -inf: a pass's single block, or block B missing)
            const float mn0 = fmaxf(m0, bm0), mn1 = fmaxf(m1, bm1);
            const float al0 = mn0 == neg_inf() ? 1.f : ex2(m0 - mn0);
            const float al1 = mn1 == neg_inf() ? 1.f : ex2(m1 - mn1);
            l0 *= al0;
            l1 *= al1;
#pragma unroll
            for (int gi = 0; gi < NG; ++gi) {
                corr[gi][0] *= al0;
                corr[gi][1] *= al1;
            }
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                o[mt][0] *= al0;
                o[mt][1] *= al1;
                o[mt][2] *= al0;
                o[mt][3] *= al1;
            }
            m0 = mn0;
            m1 = mn1;
        }
        const float r0 = m0 == neg_inf() ? 0.f : m0, r1 = m1 == neg_inf() ? 0.f : m1;
        const float p0 = ex2(x0 - r0), p1 = ex2(x1 - r1);
        const float p2 = ex2(x2 - r0), p3 = ex2(x3 - r1);
        l0 += p0 + p2;
        l1 += p1 + p3;
        const bool w0 = ok0 && !sk0, w1 = ok1 && !sk1;
        // PV weight fragments, split by column half: block A's MMAs take
        // columns 0-3 (lanes g < 4 after the transpose), block B's 4-7
        uint32_t wa0[NG], wa1[NG], wb0[NG], wb1[NG];
#pragma unroll
        for (int gi = 0; gi < NG; ++gi) {
            const float vs0 = __low2float(S.vs[gi]), vs1 = __high2float(S.vs[gi]);
            const float W0 = w0 ? p0 * vs0 : 0.f, W1 = w0 ? p1 * vs0 : 0.f;
            const float W2 = w1 ? p2 * vs1 : 0.f, W3 = w1 ? p3 * vs1 : 0.f;
            const uint32_t pk0 = f16pair(W0, W1), pk1 = f16pair(W2, W3);
            const float vz0 = __low2float(S.vz[gi]), vz1 = __high2float(S.vz[gi]);
            // masked tokens carry W = 0, but their zero point may be any
            // bits (slots never written): it is selected away, not multiplied
            const float zm0 = w0 ? vz0 : 0.f, zm1 = w1 ? vz1 : 0.f;
            const __half2 h0 = *reinterpret_cast<const __half2*>(&pk0);
            const __half2 h1 = *reinterpret_cast<const __half2*>(&pk1);
            corr[gi][0] += __low2float(h0) * zm0 + __low2float(h1) * zm1;
            corr[gi][1] += __high2float(h0) * zm0 + __high2float(h1) * zm1;
            const uint32_t t0w = movmatrix_trans(pk0), t1w = movmatrix_trans(pk1);
            wa0[gi] = g < 4 ? t0w : 0u;
            wa1[gi] = g < 4 ? t1w : 0u;
            wb0[gi] = g < 4 ? 0u : t0w;
            wb1[gi] = g < 4 ? 0u : t1w;
        }
        // ---- O^T += C_v^T W^T for both blocks (INT4 codes decode to finite
        // values, so rows past the context need no clearing: their W is 0)
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            const int el = pv_e<NG, MT>(mt, 0), eh = pv_e<NG, MT>(mt, 1);
            const int gi = (el >> 3) / VPG;
            mma_f16(o[mt], pv_frag(CA, el, 0), pv_frag(CA, eh, 0), pv_frag(CA, el, 1), pv_frag(CA, eh, 1),
                    wa0[gi], wa1[gi]);
            mma_f16(o[mt], pv_frag(CB, el, 0), pv_frag(CB, eh, 0), pv_frag(CB, el, 1), pv_frag(CB, eh, 1),
                    wb0[gi], wb1[gi]);
        }
        if (sinks_here) {
            // add P_t * sink_v[t] for the sink positions (block A's lanes)
            const T* svb = static_cast<const T*>(a.sink_v);
            for (int t = 0; t < a.n_sink && t < ctx; ++t) {
                const int src = (t & 7) * 4 + c;
                const float pa = __shfl_sync(0xffffffffu, t < 8 ? p0 : p2, src);
                const float pb = __shfl_sync(0xffffffffu, t < 8 ? p1 : p3, src);
                if (sl != 0) continue;
                const T* vrow = svb + ((static_cast<int64_t>(b) * a.n_sink + t) * a.hkv + kvh) * D;
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    const int el = pv_e<NG, MT>(mt, 0), eh = pv_e<NG, MT>(mt, 1);
                    const float u = (el & 1) ? 16.f * kInvTwo24 : kInvTwo24;
                    const float vl = tofloat(vrow[pv_column<NG, D>(el, g)]) * u;
                    const float vh = tofloat(vrow[pv_column<NG, D>(eh, g)]) * u;
                    o[mt][0] += pa * vl;
                    o[mt][1] += pb * vl;
                    o[mt][2] += pa * vh;
                    o[mt][3] += pb * vh;
                }
            }
        }
    };

    // ---- the quantised blocks, two per step
    const int qlim = WIN ? min(lb_end, win_lb0) : lb_end;
    const int nq = qlim > lb_first ? (qlim - lb_first + stride - 1) / stride : 0;
    int tab = 0;
    // Step k (blocks 2k, 2k + 1 of the pass): the physical ids its loads
    // read -- a missing or bad block reads the other one's bytes, or block
    // 0's (finite, masked) -- and its validity bits (1: A, 2: B).  The
    // table window of 32 entries is refilled at multiples of 32 blocks; a
    // step's two entries never straddle a refill.
    auto step_ids = [&](int k, int& pA, int& pB) {
        const int i = 2 * k;
        if ((i & 31) == 0) {
            const int idx = lb_first + stride * (i + lane);
            tab = idx < lb_end ? trow[idx] : -1;
        }
        const int physA = __shfl_sync(0xffffffffu, tab, i & 31);
        const int physB = __shfl_sync(0xffffffffu, tab, (i + 1) & 31);
        const bool hasB = i + 1 < nq;
        const bool vA = static_cast<unsigned>(physA) < static_cast<unsigned>(a.num_blocks);
        const bool vB = hasB && static_cast<unsigned>(physB) < static_cast<unsigned>(a.num_blocks);
        if (lane == 0 && (!vA || (hasB && !vB))) atomicOr(a.status, PKV_STATUS_BAD_BLOCK);
        pA = vA ? physA : (vB ? physB : 0);
        pB = vB ? physB : pA;
        return (vA ? 1 : 0) | (vB ? 2 : 0);
    };
    const int nsteps = (nq + 1) / 2;
    for (int k = 0; k < nsteps; ++k) {
        int pA, pB;
        const int f = step_ids(k, pA, pB);
        if (!f) continue;
        Codes CA, CB;
        Scales S;
        load_codes(pA, CA);
        load_codes(pB, CB);
        load_scales(sl ? pB : pA, S);
        attend_pair(lb_first + 2 * k * stride, (f & 1) != 0, (f & 2) != 0, CA, CB, S);
    }

    // ---- merge the two column halves: lane c (< 2) and lane c + 2 hold the
    // same query heads, token lanes and output columns for blocks A and B;
    // after the exchange both hold the merged state (lanes c >= 2 then stand
    // for the padding heads 4-7, as in the single-block layout)
    {
        const float pm0 = __shfl_xor_sync(0xffffffffu, m0, 2), pm1 = __shfl_xor_sync(0xffffffffu, m1, 2);
        const float M0 = fmaxf(m0, pm0), M1 = fmaxf(m1, pm1);
        const bool e0 = M0 == neg_inf(), e1 = M1 == neg_inf();
        const float sa0 = e0 ? 0.f : ex2(m0 - M0), sb0 = e0 ? 0.f : ex2(pm0 - M0);
        const float sa1 = e1 ? 0.f : ex2(m1 - M1), sb1 = e1 ? 0.f : ex2(pm1 - M1);
        const float pl0 = __shfl_xor_sync(0xffffffffu, l0, 2), pl1 = __shfl_xor_sync(0xffffffffu, l1, 2);
        l0 = l0 * sa0 + pl0 * sb0;
        l1 = l1 * sa1 + pl1 * sb1;
#pragma unroll
        for (int gi = 0; gi < NG; ++gi) {
            const float pc0 = __shfl_xor_sync(0xffffffffu, corr[gi][0], 2);
            const float pc1 = __shfl_xor_sync(0xffffffffu, corr[gi][1], 2);
            corr[gi][0] = corr[gi][0] * sa0 + pc0 * sb0;
            corr[gi][1] = corr[gi][1] * sa1 + pc1 * sb1;
        }
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            const float q0 = __shfl_xor_sync(0xffffffffu, o[mt][0], 2);
            const float q1 = __shfl_xor_sync(0xffffffffu, o[mt][1], 2);
            const float q2 = __shfl_xor_sync(0xffffffffu, o[mt][2], 2);
            const float q3 = __shfl_xor_sync(0xffffffffu, o[mt][3], 2);
            o[mt][0] = o[mt][0] * sa0 + q0 * sb0;
            o[mt][1] = o[mt][1] * sa1 + q1 * sb1;
            o[mt][2] = o[mt][2] * sa0 + q2 * sb0;
            o[mt][3] = o[mt][3] * sa1 + q3 * sb1;
        }
        m0 = M0;
        m1 = M1;
    }
    // ---- the 16-bit window blocks (the pass's last ones), one at a time
    if constexpr (WIN) {
        for (int lb = lb_first + nq * stride; lb < lb_end; lb += stride) attend16(lb);
    }
}

// One warp's pass over the blocks lb_first, lb_first + stride, ... < lb_end
// of sequence b, KV head kvh (context ctx): query fragments, then every block
// loaded into registers and attended into st (reset first).  sq is the
// lane's slot of the warp's shared query slice (row t at sq[t * 32]).
//
// PAIR (INT4, G <= 4): two blocks per step, one in each half of the MMA's
// eight query columns.  The GQA group fills at most four of them, so block A
// takes columns 0-3 and block B columns 4-7: its QK^T MMAs see the query in
// columns 4-7 and zeros in 0-3 (and A's the other way round), both add into
// one accumulator, and every lane's four logits are live -- lanes c = 0, 1
// hold block A's (tokens g, g + 8; heads 2c, 2c + 1), lanes c = 2, 3 block
// B's.  The whole scalar part of a step (scales, zero points, softmax, PV
// weights) then runs once for two blocks.  The two halves are two
// independent online softmaxes (even and odd blocks of the pass), each PV
// weight fragment is split by its column half into one MMA per block, and
// the halves are merged (log-sum-exp) before the window blocks and at the
// end.  The query slice holds two copies: columns 0-3 live (stream A) and
// columns 4-7 live (stream B), row t of copy s at sq[(s KSTEPS / 2 + t) 32].
template <typename T, int D, int QMODE, int NG, bool WIN, bool PAIR = false>
__device__ __forceinline__ void quant_pass(const QDecodeArgs& a, int b, int kvh, int ctx, int lb_first,
                                           int lb_end, int stride, uint4* sq, QState<D / 16, NG>& st) {
    constexpr bool INT4 = QMODE == PKV_QMODE_INT4_ASYM;
    constexpr int KSTEPS = D / 16;             // k-steps of QK^T
    constexpr int MT = D / 16;                 // m-tiles of PV
    constexpr int CB = INT4 ? D / 2 : D;       // code bytes per row
    constexpr int KW = INT4 ? D / 32 : D / 16; // 32-bit K-code words per lane per row
    constexpr int VW = INT4 ? D / 64 : D / 32; // 32-bit V-code words per lane per row
    constexpr int DS = D / 8;                  // head-dim columns per lane group in PV
    // INT4 column groups (one (scale, zero) each): GS columns, KPG K words
    // and VPG V words per lane and row in each
    constexpr int GS = D / NG;
    constexpr int KPG = KW / NG;
    constexpr int VPG = VW / NG;
    static_assert(NG == 1 || (INT4 && D == 128 && NG == 2), "groups: one per head, or 64 columns at D 128");
    static_assert(!PAIR || INT4, "paired blocks: INT4 only");
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
    // hh: the lane's S / O columns are query heads 2 hh, 2 hh + 1 (of its
    // stream when PAIR); qh: the query head whose B-fragment column it feeds
    const int hh = PAIR ? (c & 1) : c;
    const int qh = PAIR ? (g & 3) : g;

    // ---- query fragments (fp16) in the permuted k order of the code layout
    // staged in this warp's shared slice (k-steps 2t, 2t + 1 of lane l at
    // sq[warp][t][l]) and re-read per block, to leave registers for the codes
    uint32_t qf[KSTEPS][2];
    float qsum[NG];  // sums over this lane's columns of query head g, per group
#pragma unroll
    for (int gi = 0; gi < NG; ++gi) qsum[gi] = 0.f;
    {
        const T* qrow = static_cast<const T*>(a.q) +
                        (static_cast<int64_t>(b) * a.hq + kvh * a.G + (qh < a.G ? qh : 0)) * D;
        const bool valid = qh < a.G;
        if constexpr (INT4) {
            // K word k of lane c covers the 8 columns starting at
            // (k / KPG) GS + (GS / 4) c + 8 (k % KPG): lane c holds a quarter
            // of every column group
#pragma unroll
            for (int k = 0; k < KW; ++k) {
                const int col = (k / KPG) * GS + (GS / 4) * c + 8 * (k % KPG);
                float x[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) x[j] = valid ? tofloat(qrow[col + j]) : 0.f;
                // fp16 rounding of the query, as fed to the MMA
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    x[j] = __half2float(__float2half_rn(x[j]));
                    qsum[k / KPG] += x[j];
                }
                // the odd nibbles enter the MMA 16x larger: their query
                // columns go in divided by 16 (a power of two)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    qf[2 * k + e][0] = f16pair(x[2 * e], x[2 * e + 4]);
                    qf[2 * k + e][1] = f16pair(x[2 * e + 1] * 0.0625f, x[2 * e + 5] * 0.0625f);
                }
            }
        } else {
            // load i covers columns [64i + 16c, +16), four k-steps
#pragma unroll
            for (int i = 0; i < D / 64; ++i) {
                float x[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) x[j] = valid ? tofloat(qrow[64 * i + 16 * c + j]) : 0.f;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    qf[4 * i + e][0] = f16pair(x[4 * e], x[4 * e + 1]);
                    qf[4 * i + e][1] = f16pair(x[4 * e + 2], x[4 * e + 3]);
                }
            }
        }
    }
    // full per-head sums: reduce over the 4 lanes of head g, then fetch the
    // sums of this lane's PV/S columns (heads 2c, 2c+1)
    __syncwarp();  // the previous pass no longer reads the slice
    if constexpr (kQueryInShared<QMODE>) {
#pragma unroll
        for (int t = 0; t < KSTEPS / 2; ++t) {
            const uint4 v = make_uint4(qf[2 * t][0], qf[2 * t][1], qf[2 * t + 1][0], qf[2 * t + 1][1]);
            if constexpr (PAIR) {
                const uint4 z = make_uint4(0u, 0u, 0u, 0u);
                sq[t * 32] = g < 4 ? v : z;
                sq[(KSTEPS / 2 + t) * 32] = g < 4 ? z : v;
            } else {
                sq[t * 32] = v;
            }
        }
        __syncwarp();
    }
    const uint32_t qs = static_cast<uint32_t>(__cvta_generic_to_shared(sq));
    float qs0[NG], qs1[NG];  // group sums of heads 2 hh, 2 hh + 1
#pragma unroll
    for (int gi = 0; gi < NG; ++gi) {
        float x = qsum[gi];
        x += __shfl_xor_sync(0xffffffffu, x, 1);
        x += __shfl_xor_sync(0xffffffffu, x, 2);
        qs0[gi] = __shfl_sync(0xffffffffu, x, (2 * hh) * 4);
        qs1[gi] = __shfl_sync(0xffffffffu, x, (2 * hh + 1) * 4);
    }

    float& m0 = st.m0;
    float& m1 = st.m1;
    float& l0 = st.l0;
    float& l1 = st.l1;
    auto& corr = st.corr;
    auto& o = st.o;
    st.init();

    const int32_t* trow = a.tables + static_cast<int64_t>(b) * a.max_blocks;
    const int vr0 = 2 * c, vr1 = 2 * c + 1, vr2 = 8 + 2 * c, vr3 = 9 + 2 * c;

    // One block's codes and per-token (scale, zero) for this lane.
    struct QBlk {
        uint32_t kw0[KW], kw1[KW], vw[4][VW];
        __half2 ks[NG], vs[NG], kz[NG], vz[NG];  // per group; low: token g, high: token g + 8
    };
    auto load = [&](int phys, QBlk& B) {
        const int64_t bh = static_cast<int64_t>(phys) * a.hkv + kvh;  // (block, head)
        const uint8_t* kc = a.k_codes + bh * (BS * CB);
        const uint8_t* vc = a.v_codes + bh * (BS * CB);

        // ---- loads: K rows g, g+8; V rows 2c, 2c+1, 8+2c, 9+2c; scales
        if constexpr (INT4 && NG == 2) {
            // per group: K words at byte 32 grp + 8 c, V word at byte 32 grp + 4 g
#pragma unroll
            for (int gi = 0; gi < 2; ++gi) {
                const uint2 r0 = ldg_stream8(kc + g * CB + 32 * gi + 8 * c);
                const uint2 r1 = ldg_stream8(kc + (g + 8) * CB + 32 * gi + 8 * c);
                B.kw0[2 * gi] = r0.x; B.kw0[2 * gi + 1] = r0.y;
                B.kw1[2 * gi] = r1.x; B.kw1[2 * gi + 1] = r1.y;
                const int off = 32 * gi + 4 * g;
                B.vw[0][gi] = *reinterpret_cast<const uint32_t*>(vc + vr0 * CB + off);
                B.vw[1][gi] = *reinterpret_cast<const uint32_t*>(vc + vr1 * CB + off);
                B.vw[2][gi] = *reinterpret_cast<const uint32_t*>(vc + vr2 * CB + off);
                B.vw[3][gi] = *reinterpret_cast<const uint32_t*>(vc + vr3 * CB + off);
            }
        } else if constexpr (INT4) {
            if constexpr (KW == 4) {
                const uint4 r0 = ldg_stream(kc + g * CB + 16 * c);
                const uint4 r1 = ldg_stream(kc + (g + 8) * CB + 16 * c);
                B.kw0[0] = r0.x; B.kw0[1] = r0.y; B.kw0[2] = r0.z; B.kw0[3] = r0.w;
                B.kw1[0] = r1.x; B.kw1[1] = r1.y; B.kw1[2] = r1.z; B.kw1[3] = r1.w;
            } else {
                const uint2 r0 = ldg_stream8(kc + g * CB + 8 * c);
                const uint2 r1 = ldg_stream8(kc + (g + 8) * CB + 8 * c);
                B.kw0[0] = r0.x; B.kw0[1] = r0.y;
                B.kw1[0] = r1.x; B.kw1[1] = r1.y;
            }
            if constexpr (VW == 2) {
                const int off = DS / 2 * g;  // bytes: DS columns = DS/2 bytes
                const uint2 x0 = ldg_stream8(vc + vr0 * CB + off), x1 = ldg_stream8(vc + vr1 * CB + off);
                const uint2 x2 = ldg_stream8(vc + vr2 * CB + off), x3 = ldg_stream8(vc + vr3 * CB + off);
                B.vw[0][0] = x0.x; B.vw[0][1] = x0.y; B.vw[1][0] = x1.x; B.vw[1][1] = x1.y;
                B.vw[2][0] = x2.x; B.vw[2][1] = x2.y; B.vw[3][0] = x3.x; B.vw[3][1] = x3.y;
            } else {
                const int off = DS / 2 * g;
                B.vw[0][0] = *reinterpret_cast<const uint32_t*>(vc + vr0 * CB + off);
                B.vw[1][0] = *reinterpret_cast<const uint32_t*>(vc + vr1 * CB + off);
                B.vw[2][0] = *reinterpret_cast<const uint32_t*>(vc + vr2 * CB + off);
                B.vw[3][0] = *reinterpret_cast<const uint32_t*>(vc + vr3 * CB + off);
            }
        } else {
#pragma unroll
            for (int i = 0; i < D / 64; ++i) {
                const uint4 r0 = ldg_stream(kc + g * CB + 64 * i + 16 * c);
                const uint4 r1 = ldg_stream(kc + (g + 8) * CB + 64 * i + 16 * c);
                B.kw0[4 * i] = r0.x; B.kw0[4 * i + 1] = r0.y; B.kw0[4 * i + 2] = r0.z; B.kw0[4 * i + 3] = r0.w;
                B.kw1[4 * i] = r1.x; B.kw1[4 * i + 1] = r1.y; B.kw1[4 * i + 2] = r1.z; B.kw1[4 * i + 3] = r1.w;
            }
            const int off = DS * g;  // bytes
            if constexpr (VW == 4) {
                const uint4 x0 = ldg_stream(vc + vr0 * CB + off), x1 = ldg_stream(vc + vr1 * CB + off);
                const uint4 x2 = ldg_stream(vc + vr2 * CB + off), x3 = ldg_stream(vc + vr3 * CB + off);
                B.vw[0][0] = x0.x; B.vw[0][1] = x0.y; B.vw[0][2] = x0.z; B.vw[0][3] = x0.w;
                B.vw[1][0] = x1.x; B.vw[1][1] = x1.y; B.vw[1][2] = x1.z; B.vw[1][3] = x1.w;
                B.vw[2][0] = x2.x; B.vw[2][1] = x2.y; B.vw[2][2] = x2.z; B.vw[2][3] = x2.w;
                B.vw[3][0] = x3.x; B.vw[3][1] = x3.y; B.vw[3][2] = x3.z; B.vw[3][3] = x3.w;
            } else {
                const uint2 x0 = ldg_stream8(vc + vr0 * CB + off), x1 = ldg_stream8(vc + vr1 * CB + off);
                const uint2 x2 = ldg_stream8(vc + vr2 * CB + off), x3 = ldg_stream8(vc + vr3 * CB + off);
                B.vw[0][0] = x0.x; B.vw[0][1] = x0.y; B.vw[1][0] = x1.x; B.vw[1][1] = x1.y;
                B.vw[2][0] = x2.x; B.vw[2][1] = x2.y; B.vw[3][0] = x3.x; B.vw[3][1] = x3.y;
            }
        }
        // scale / zero [block, head, token, group]
        const int64_t s0 = (bh * BS + g) * NG, s1 = (bh * BS + g + 8) * NG;
#pragma unroll
        for (int gi = 0; gi < NG; ++gi) {
            B.ks[gi] = __halves2half2(a.k_scale[s0 + gi], a.k_scale[s1 + gi]);
            B.vs[gi] = __halves2half2(a.v_scale[s0 + gi], a.v_scale[s1 + gi]);
            if constexpr (INT4) {
                B.kz[gi] = __halves2half2(a.k_zero[s0 + gi], a.k_zero[s1 + gi]);
                B.vz[gi] = __halves2half2(a.v_zero[s0 + gi], a.v_zero[s1 + gi]);
            }
        }
    };
    auto attend = [&](int lb, QBlk& B) {
        // ---- S_raw^T = C Q^T over the code values (INT4: one accumulator per group)
        float sg[NG][4];
#pragma unroll
        for (int gi = 0; gi < NG; ++gi) sg[gi][0] = sg[gi][1] = sg[gi][2] = sg[gi][3] = 0.f;
        float (&s)[4] = sg[0];
        if constexpr (INT4) {
#pragma unroll
            for (int k = 0; k < KW; ++k) {
                // k-step 2k: nibbles {0, 4} and {1, 5}; 2k + 1: {2, 6}, {3, 7}
                const uint4 q2 = kQueryInShared<QMODE> ? lds128(qs + k * 512)
                                      : make_uint4(qf[2 * k][0], qf[2 * k][1], qf[2 * k + 1][0], qf[2 * k + 1][1]);
                const uint32_t u0 = B.kw0[k] >> 8, u1 = B.kw1[k] >> 8;
                float (&sk)[4] = sg[k / KPG];
                mma_f16(sk, nib_even(B.kw0[k]), nib_even(B.kw1[k]), nib_odd(B.kw0[k]), nib_odd(B.kw1[k]),
                        q2.x, q2.y);
                mma_f16(sk, nib_even(u0), nib_even(u1), nib_odd(u0), nib_odd(u1), q2.z, q2.w);
            }
        } else {
#pragma unroll
            for (int t = 0; t < KSTEPS / 2; ++t) {
                // k-step j = 4i + e uses word e of load i (= word j): codes
                // {0, 1} are the low k pair, codes {2, 3} the high k pair
                const int j0 = 2 * t, j1 = 2 * t + 1;
                const uint4 q2 = kQueryInShared<QMODE> ? lds128(qs + t * 512)
                                      : make_uint4(qf[j0][0], qf[j0][1], qf[j1][0], qf[j1][1]);
                mma_f16(s, e4m3x2(B.kw0[j0]), e4m3x2(B.kw1[j0]), e4m3x2(B.kw0[j0] >> 16),
                        e4m3x2(B.kw1[j0] >> 16), q2.x, q2.y);
                mma_f16(s, e4m3x2(B.kw0[j1]), e4m3x2(B.kw1[j1]), e4m3x2(B.kw0[j1] >> 16),
                        e4m3x2(B.kw1[j1] >> 16), q2.z, q2.w);
            }
        }
        const int t0 = lb * BS;
        const int tok0 = t0 + g;
        const bool ok0 = tok0 < ctx, ok1 = tok0 + 8 < ctx;
        float x0, x1, x2, x3;
        if constexpr (INT4) {
            // S = sum_groups s (sum_d q_d c_d - z sum_d q_d); the MMA gave
            // 2^-24 sum q c per group
            x0 = x1 = x2 = x3 = 0.f;
#pragma unroll
            for (int gi = 0; gi < NG; ++gi) {
                const float ks0 = __low2float(B.ks[gi]), ks1 = __high2float(B.ks[gi]);
                const float kz0 = __low2float(B.kz[gi]), kz1 = __high2float(B.kz[gi]);
                x0 += ks0 * (sg[gi][0] * kTwo24 - kz0 * qs0[gi]);
                x1 += ks0 * (sg[gi][1] * kTwo24 - kz0 * qs1[gi]);
                x2 += ks1 * (sg[gi][2] * kTwo24 - kz1 * qs0[gi]);
                x3 += ks1 * (sg[gi][3] * kTwo24 - kz1 * qs1[gi]);
            }
            x0 *= a.scale_log2;
            x1 *= a.scale_log2;
            x2 *= a.scale_log2;
            x3 *= a.scale_log2;
        } else {
            const float ks0 = __low2float(B.ks[0]), ks1 = __high2float(B.ks[0]);
            x0 = ks0 * s[0] * a.scale_log2;
            x1 = ks0 * s[1] * a.scale_log2;
            x2 = ks1 * s[2] * a.scale_log2;
            x3 = ks1 * s[3] * a.scale_log2;
        }
        const bool sinks_here = lb == 0 && a.n_sink > 0;
        bool sk0 = false, sk1 = false;
        if (sinks_here) {
            // exact 16-bit sink keys for positions < n_sink
            sk0 = g < a.n_sink;
            sk1 = g + 8 < a.n_sink;
            const T* qbase = static_cast<const T*>(a.q) + (static_cast<int64_t>(b) * a.hq + kvh * a.G) * D;
            const T* skb = static_cast<const T*>(a.sink_k);
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int t = g + 8 * r;
                if (t < a.n_sink) {
                    const T* krow = skb + ((static_cast<int64_t>(b) * a.n_sink + t) * a.hkv + kvh) * D;
                    float d0 = 0.f, d1 = 0.f;
                    const int h0 = min(2 * hh, a.G - 1), h1 = min(2 * hh + 1, a.G - 1);
                    for (int d = 0; d < D; ++d) {
                        const float kv = tofloat(krow[d]);
                        d0 += tofloat(qbase[h0 * D + d]) * kv;
                        d1 += tofloat(qbase[h1 * D + d]) * kv;
                    }
                    if (r == 0) {
                        x0 = d0 * a.scale_log2;
                        x1 = d1 * a.scale_log2;
                    } else {
                        x2 = d0 * a.scale_log2;
                        x3 = d1 * a.scale_log2;
                    }
                }
            }
        }
        if (!ok0) x0 = x1 = neg_inf();
        if (!ok1) x2 = x3 = neg_inf();

        // ---- online softmax (base 2).  The reference max m is raised only
        // when a logit of the block exceeds it by more than kSlack; otherwise
        // the weights 2^(x - m) <= 2^kSlack are taken against the old m, with
        // no warp-wide max and no rescale (m cancels in o / l and the merges).
        // A block whose V scales could carry W = P s past the fp16 range at
        // P = 2^kSlack takes the exact max (then P <= 1, W <= s).
        const float bx0 = fmaxf(x0, x2), bx1 = fmaxf(x1, x3);
        float vsmax = 0.f;
#pragma unroll
        for (int gi = 0; gi < NG; ++gi)
            vsmax = fmaxf(vsmax, fmaxf(__low2float(B.vs[gi]), __high2float(B.vs[gi])));
        if (__any_sync(0xffffffffu, bx0 > m0 + kSlack || bx1 > m1 + kSlack || vsmax > kLazyMaxScale)) {
            float bm0 = bx0, bm1 = bx1;
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                bm0 = fmaxf(bm0, __shfl_xor_sync(0xffffffffu, bm0, off));
                bm1 = fmaxf(bm1, __shfl_xor_sync(0xffffffffu, bm1, off));
            }
            const float mn0 = fmaxf(m0, bm0), mn1 = fmaxf(m1, bm1);
            const float al0 = ex2(m0 - mn0), al1 = ex2(m1 - mn1);
            l0 *= al0;
            l1 *= al1;
#pragma unroll
            for (int gi = 0; gi < NG; ++gi) {
                corr[gi][0] *= al0;
                corr[gi][1] *= al1;
            }
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                o[mt][0] *= al0;
                o[mt][1] *= al1;
                o[mt][2] *= al0;
                o[mt][3] *= al1;
            }
            m0 = mn0;
            m1 = mn1;
        }
        const float p0 = ex2(x0 - m0), p1 = ex2(x1 - m1);
        const float p2 = ex2(x2 - m0), p3 = ex2(x3 - m1);
        l0 += p0 + p2;
        l1 += p1 + p3;
        // PV weights W = P * s per group (zero for masked and sink tokens)
        const bool w0 = ok0 && !sk0, w1 = ok1 && !sk1;
        uint32_t pb0[NG], pb1[NG];
#pragma unroll
        for (int gi = 0; gi < NG; ++gi) {
            const float vs0 = __low2float(B.vs[gi]), vs1 = __high2float(B.vs[gi]);
            const float W0 = w0 ? p0 * vs0 : 0.f, W1 = w0 ? p1 * vs0 : 0.f;
            const float W2 = w1 ? p2 * vs1 : 0.f, W3 = w1 ? p3 * vs1 : 0.f;
            const uint32_t pk0 = f16pair(W0, W1), pk1 = f16pair(W2, W3);
            if constexpr (INT4) {
                // the correction uses the fp16-rounded weights the MMA sees
                const float vz0 = __low2float(B.vz[gi]), vz1 = __high2float(B.vz[gi]);
                const __half2 h0 = *reinterpret_cast<const __half2*>(&pk0);
                const __half2 h1 = *reinterpret_cast<const __half2*>(&pk1);
                if (w0) {
                    corr[gi][0] += __low2float(h0) * vz0;
                    corr[gi][1] += __high2float(h0) * vz0;
                }
                if (w1) {
                    corr[gi][0] += __low2float(h1) * vz1;
                    corr[gi][1] += __high2float(h1) * vz1;
                }
            }
            pb0[gi] = movmatrix_trans(pk0);
            pb1[gi] = movmatrix_trans(pk1);
        }

        if (t0 + BS > ctx) {  // partial last block: clear codes of missing tokens
#pragma unroll
            for (int j = 0; j < VW; ++j) {
                if (t0 + vr0 >= ctx) B.vw[0][j] = 0;
                if (t0 + vr1 >= ctx) B.vw[1][j] = 0;
                if (t0 + vr2 >= ctx) B.vw[2][j] = 0;
                if (t0 + vr3 >= ctx) B.vw[3][j] = 0;
            }
        }

        // ---- O^T += C_v^T W^T: m-tile mt takes the lane's elements
        // e = pv_e<NG>(mt, 0 / 1) (see pv_e), both in one column group
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            uint32_t av[4];
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const int e = INT4 ? pv_e<NG, MT>(mt, hf) : mt + hf * MT;
#pragma unroll
                for (int pr = 0; pr < 2; ++pr) {  // token pair (2c, 2c+1) / (8+2c, 9+2c)
                    const uint32_t* R0 = B.vw[2 * pr];
                    const uint32_t* R1 = B.vw[2 * pr + 1];
                    uint32_t v;
                    if constexpr (INT4) {
                        const int word = e >> 3, sub = (e >> 2) & 1, nib = e & 3;
                        const uint32_t X = __byte_perm(R0[word], R1[word], sub ? 0x7632u : 0x5410u);
                        const uint32_t Y = nib >= 2 ? X >> 8 : X;
                        v = (nib & 1) ? nib_odd(Y) : nib_even(Y);
                    } else {
                        const int word = e >> 2, sub = e & 3;
                        const uint32_t X = __byte_perm(R0[word], R1[word], (sub >> 1) ? 0x7362u : 0x5140u);
                        v = e4m3x2((sub & 1) ? (X >> 16) : X);
                    }
                    av[hf + 2 * pr] = v;
                }
            }
            const int gi = INT4 ? (pv_e<NG, MT>(mt, 0) >> 3) / VPG : 0;
            mma_f16(o[mt], av[0], av[1], av[2], av[3], pb0[gi], pb1[gi]);
        }

        if (sinks_here) {
            // add P_t * sink_v[t] for the sink positions, in fp32
            const T* svb = static_cast<const T*>(a.sink_v);
            for (int t = 0; t < a.n_sink && t < ctx; ++t) {
                const int src = (t & 7) * 4 + c;
                const float pa = __shfl_sync(0xffffffffu, t < 8 ? p0 : p2, src);
                const float pb = __shfl_sync(0xffffffffu, t < 8 ? p1 : p3, src);
                const T* vrow = svb + ((static_cast<int64_t>(b) * a.n_sink + t) * a.hkv + kvh) * D;
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    // in the accumulator's units (INT4: 2^-24, odd columns 2^-20)
                    const int el = INT4 ? pv_e<NG, MT>(mt, 0) : mt, eh = INT4 ? pv_e<NG, MT>(mt, 1) : mt + MT;
                    const float u = INT4 ? ((el & 1) ? 16.f * kInvTwo24 : kInvTwo24) : 1.f;
                    const float vl = tofloat(vrow[pv_column<INT4 ? NG : 1, D>(el, g)]) * u;
                    const float vh = tofloat(vrow[pv_column<INT4 ? NG : 1, D>(eh, g)]) * u;
                    o[mt][0] += pa * vl;
                    o[mt][1] += pb * vl;
                    o[mt][2] += pa * vh;
                    o[mt][3] += pb * vh;
                }
            }
        }
    };

    // ---- 16-bit window blocks (the run's last blocks): read from the ring
    // in the 16-bit decode layout, accumulated into o in true units (o is
    // converted once, before the first of them; they come after every
    // quantised block of the pass)
    auto attend16 = [&](int lb) {
        using H = Half16<T>;
        constexpr int KC = D / 32;
        constexpr int VC = D / 64;
        if (!st.true_units) {
            // the correction is a per-lane partial sum: total it over the 8
            // token lanes first
#pragma unroll
            for (int gi = 0; gi < NG; ++gi) {
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) {
                    corr[gi][0] += __shfl_xor_sync(0xffffffffu, corr[gi][0], off);
                    corr[gi][1] += __shfl_xor_sync(0xffffffffu, corr[gi][1], off);
                }
            }
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                const int el = INT4 ? pv_e<NG, MT>(mt, 0) : mt;
                const int gi = INT4 ? (el >> 3) / VPG : 0;
                const float u = INT4 ? ((el & 1) ? kTwo24 * 0.0625f : kTwo24) : 1.f;
                o[mt][0] = o[mt][0] * u - corr[gi][0];
                o[mt][1] = o[mt][1] * u - corr[gi][1];
                o[mt][2] = o[mt][2] * u - corr[gi][0];
                o[mt][3] = o[mt][3] * u - corr[gi][1];
            }
#pragma unroll
            for (int gi = 0; gi < NG; ++gi) corr[gi][0] = corr[gi][1] = 0.f;
            st.true_units = true;
        }
        const int64_t rbase = ((static_cast<int64_t>(b) * a.ring + lb % a.ring) * a.hkv + kvh) * (BS * D);
        const T* wk = static_cast<const T*>(a.win_k) + rbase;
        const T* wv = static_cast<const T*>(a.win_v) + rbase;
        // QK^T: K rows g, g+8 and query head g at [32i + 8c, +8)
        float s4[4] = {0.f, 0.f, 0.f, 0.f};
        {
            const T* qrow = static_cast<const T*>(a.q) +
                            (static_cast<int64_t>(b) * a.hq + kvh * a.G + (g < a.G ? g : 0)) * D;
            uint4 k0[KC], k1[KC], qv[KC];
#pragma unroll
            for (int i = 0; i < KC; ++i) {
                k0[i] = ldg_stream(wk + g * D + 32 * i + 8 * c);
                k1[i] = ldg_stream(wk + (g + 8) * D + 32 * i + 8 * c);
                qv[i] = g < a.G ? *reinterpret_cast<const uint4*>(qrow + 32 * i + 8 * c) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int i = 0; i < KC; ++i) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    H::mma(s4, word(k0[i], 2 * e), word(k1[i], 2 * e), word(k0[i], 2 * e + 1),
                           word(k1[i], 2 * e + 1), word(qv[i], 2 * e), word(qv[i], 2 * e + 1));
                }
            }
        }
        const int t0 = lb * BS;
        const bool ok0 = t0 + g < ctx, ok1 = t0 + g + 8 < ctx;
        const float x0 = ok0 ? s4[0] * a.scale_log2 : neg_inf();
        const float x1 = ok0 ? s4[1] * a.scale_log2 : neg_inf();
        const float x2 = ok1 ? s4[2] * a.scale_log2 : neg_inf();
        const float x3 = ok1 ? s4[3] * a.scale_log2 : neg_inf();
        float bm0 = fmaxf(x0, x2), bm1 = fmaxf(x1, x3);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            bm0 = fmaxf(bm0, __shfl_xor_sync(0xffffffffu, bm0, off));
            bm1 = fmaxf(bm1, __shfl_xor_sync(0xffffffffu, bm1, off));
        }
        const float mn0 = fmaxf(m0, bm0), mn1 = fmaxf(m1, bm1);
        if (mn0 != m0 || mn1 != m1) {
            const float al0 = ex2(m0 - mn0), al1 = ex2(m1 - mn1);
            l0 *= al0;
            l1 *= al1;
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                o[mt][0] *= al0;
                o[mt][1] *= al1;
                o[mt][2] *= al0;
                o[mt][3] *= al1;
            }
            m0 = mn0;
            m1 = mn1;
        }
        const float p0 = ex2(x0 - m0), p1 = ex2(x1 - m1);
        const float p2 = ex2(x2 - m0), p3 = ex2(x3 - m1);
        l0 += p0 + p2;
        l1 += p1 + p3;
        const uint32_t h01 = H::pack(p0, p1), h23 = H::pack(p2, p3);
        const uint32_t pb0 = movmatrix_trans(h01), pb1 = movmatrix_trans(h23);
        uint32_t pr0 = 0, pr1 = 0;
        constexpr bool kSplit = sizeof(T) == 2 && !std::is_same<T, __half>::value;  // bf16 P: value + residual
        if constexpr (kSplit) {
            pr0 = movmatrix_trans(H::pack(p0 - __uint_as_float(h01 << 16), p1 - __uint_as_float(h01 & 0xffff0000u)));
            pr1 = movmatrix_trans(H::pack(p2 - __uint_as_float(h23 << 16), p3 - __uint_as_float(h23 & 0xffff0000u)));
        }
        // PV: V rows 2c, 2c+1, 8+2c, 9+2c at the lane's columns (chunk j: the 8
        // columns from pv_column(8 j, g)), rows past the context cleared
        uint4 vv[4][VC];
#pragma unroll
        for (int j = 0; j < VC; ++j) {
            const int col = pv_column<INT4 ? NG : 1, D>(8 * j, g);
            vv[0][j] = ldg_stream(wv + (2 * c) * D + col);
            vv[1][j] = ldg_stream(wv + (2 * c + 1) * D + col);
            vv[2][j] = ldg_stream(wv + (8 + 2 * c) * D + col);
            vv[3][j] = ldg_stream(wv + (9 + 2 * c) * D + col);
            if (t0 + 2 * c >= ctx) vv[0][j] = make_uint4(0, 0, 0, 0);
            if (t0 + 2 * c + 1 >= ctx) vv[1][j] = make_uint4(0, 0, 0, 0);
            if (t0 + 8 + 2 * c >= ctx) vv[2][j] = make_uint4(0, 0, 0, 0);
            if (t0 + 9 + 2 * c >= ctx) vv[3][j] = make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            const int el = INT4 ? pv_e<NG, MT>(mt, 0) : mt, eh = INT4 ? pv_e<NG, MT>(mt, 1) : mt + MT;
            const int jl = el >> 3, wl = (el & 7) >> 1, jh = eh >> 3, wh = (eh & 7) >> 1;
            const uint32_t sl = (el & 1) ? 0x7632u : 0x5410u, sh = (eh & 1) ? 0x7632u : 0x5410u;
            const uint32_t a0 = __byte_perm(word(vv[0][jl], wl), word(vv[1][jl], wl), sl);
            const uint32_t a1 = __byte_perm(word(vv[0][jh], wh), word(vv[1][jh], wh), sh);
            const uint32_t a2 = __byte_perm(word(vv[2][jl], wl), word(vv[3][jl], wl), sl);
            const uint32_t a3 = __byte_perm(word(vv[2][jh], wh), word(vv[3][jh], wh), sh);
            H::mma(o[mt], a0, a1, a2, a3, pb0, pb1);
            if constexpr (kSplit) H::mma(o[mt], a0, a1, a2, a3, pr0, pr1);
        }
    };

    // blocks from win_lb0 on are read from the 16-bit window ring (WIN:
    // kernels built for calls with a window; the others carry no such code)
    const int win_lb0 = WIN ? max(ctx - a.window, 0) / BS : 0x7fffffff;

    if constexpr (PAIR) {
        quant_pairs<T, D, NG, WIN>(a, b, kvh, ctx, lb_first, lb_end, stride, win_lb0, qs, qs0, qs1, st,
                                   attend16);
        return;
    }

    // Lane j holds the physical id of the pass's j-th upcoming block (32 at
    // a time), so a block's loads never wait behind a table load.
    int tab = 0;
    for (int i = 0, lb = lb_first; lb < lb_end; ++i, lb += stride) {
        if ((i & 31) == 0) {
            const int idx = lb + stride * lane;
            tab = idx < lb_end ? trow[idx] : -1;
        }
        if constexpr (WIN) {
            if (lb >= win_lb0) {
                attend16(lb);
                continue;
            }
        }
        const int phys = __shfl_sync(0xffffffffu, tab, i & 31);
        if (static_cast<unsigned>(phys) >= static_cast<unsigned>(a.num_blocks)) {
            if (lane == 0) atomicOr(a.status, PKV_STATUS_BAD_BLOCK);
            continue;
        }
        QBlk B;
        load(phys, B);
        attend(lb, B);
    }
}

// Lane-final values of a pass: l and the corrections summed over the 8
// token lanes, and the output column values sum_t W_t (c - z) in true units.
template <int D, int QMODE, int NG>
__device__ __forceinline__ void quant_finish(QState<D / 16, NG>& st) {
    constexpr bool INT4 = QMODE == PKV_QMODE_INT4_ASYM;
    constexpr int MT = D / 16;
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        st.l0 += __shfl_xor_sync(0xffffffffu, st.l0, off);
        st.l1 += __shfl_xor_sync(0xffffffffu, st.l1, off);
#pragma unroll
        for (int gi = 0; gi < NG; ++gi) {
            st.corr[gi][0] += __shfl_xor_sync(0xffffffffu, st.corr[gi][0], off);
            st.corr[gi][1] += __shfl_xor_sync(0xffffffffu, st.corr[gi][1], off);
        }
    }
    if (st.true_units) return;  // converted before the first window block
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
        // INT4: back from the accumulator's units (both elements of an m-tile
        // share their parity and column group), then O = sum W c - sum W z
        const int el = INT4 ? pv_e<NG, MT>(mt, 0) : mt;
        const int gi = INT4 ? (el >> 3) / ((D / 64) / NG) : 0;
        const float u = INT4 ? ((el & 1) ? kTwo24 * 0.0625f : kTwo24) : 1.f;
        st.o[mt][0] = st.o[mt][0] * u - st.corr[gi][0];
        st.o[mt][1] = st.o[mt][1] * u - st.corr[gi][1];
        st.o[mt][2] = st.o[mt][2] * u - st.corr[gi][0];
        st.o[mt][3] = st.o[mt][3] * u - st.corr[gi][1];
    }
}

// Shared-memory row index of the lane's output columns of m-tile mt.
template <int D, int QMODE, int NG>
__device__ __forceinline__ void out_columns(int mt, int g, int& dl, int& dh) {
    constexpr bool INT4 = QMODE == PKV_QMODE_INT4_ASYM;
    constexpr int MT = D / 16;
    const int el = INT4 ? pv_e<NG, MT>(mt, 0) : mt, eh = INT4 ? pv_e<NG, MT>(mt, 1) : mt + MT;
    dl = pv_column<INT4 ? NG : 1, D>(el, g);
    dh = pv_column<INT4 ? NG : 1, D>(eh, g);
}

// Partition kernel: one CTA of NW warps per (partition, KV head, sequence);
// the warps take the partition's blocks round-robin and merge through
// shared memory.
template <typename T, int D, int QMODE, int NG, bool WIN, bool SPLIT, bool PAIR>
__global__ void __launch_bounds__(NW * 32, kCtasPerSm<QMODE, NG, PAIR>) paged_decode_quant_kernel(QDecodeArgs a) {
    constexpr int KSTEPS = D / 16;
    constexpr int MT = D / 16;
    const int p = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, c = lane & 3;

    int ctx = a.ctx_lens[b];
    const int cap = a.max_blocks * BS;
    if (ctx < 0 || ctx > cap) {
        if (threadIdx.x == 0 && p == 0 && kvh == 0) atomicOr(a.status, PKV_STATUS_BAD_CONTEXT);
        ctx = ctx < 0 ? 0 : cap;
    }
    const int nblk = (ctx + BS - 1) / BS;
    const int nparts = (nblk + a.part_blocks - 1) / a.part_blocks;
    if (p >= (nparts > 0 ? nparts : 1)) return;
    const int blk_begin = p * a.part_blocks;
    const int blk_end = min(blk_begin + a.part_blocks, nblk);

    __shared__ uint4 sq[NW][PAIR ? 2 : 1][KSTEPS / 2][32];
    QState<MT, NG> st;
    quant_pass<T, D, QMODE, NG, WIN, PAIR>(a, b, kvh, ctx, blk_begin + warp, blk_end, NW, &sq[warp][0][0][lane],
                                           st);
    quant_finish<D, QMODE, NG>(st);
    const float m0 = st.m0, m1 = st.m1, l0 = st.l0, l1 = st.l1;
    auto& o = st.o;

    __shared__ float sm_ml[NW][8][2];
    __shared__ float sm_o[NW][8][D];
    if (g == 0) {
        sm_ml[warp][2 * c][0] = m0;
        sm_ml[warp][2 * c][1] = l0;
        sm_ml[warp][2 * c + 1][0] = m1;
        sm_ml[warp][2 * c + 1][1] = l1;
    }
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
        int dl, dh;
        out_columns<D, QMODE, NG>(mt, g, dl, dh);
        sm_o[warp][2 * c][dl] = o[mt][0];
        sm_o[warp][2 * c + 1][dl] = o[mt][1];
        sm_o[warp][2 * c][dh] = o[mt][2];
        sm_o[warp][2 * c + 1][dh] = o[mt][3];
    }
    __syncthreads();

    for (int idx = threadIdx.x; idx < a.G * D; idx += NW * 32) {
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
        const int64_t qh = static_cast<int64_t>(b) * a.hq + kvh * a.G + h;
        if constexpr (SPLIT) {
            const int64_t row = qh * a.max_parts + p;
            a.ws_o[row * D + d] = acc;
            if (d == 0) {
                a.ws_ml[2 * row] = M;
                a.ws_ml[2 * row + 1] = L;
            }
        } else {
            static_cast<T*>(a.out)[qh * D + d] = Half16<T>::from_float(L > 0.f ? acc / L : 0.f);
        }
    }
}

// Balanced split for the quantised cache (the split itself: balanced.cuh):
// warp i walks its range run by run, one pass per run segment, and writes
// the run's partial.  No barrier.
template <typename T, int D, int QMODE, int NG, bool WIN, bool PAIR>
__global__ void __launch_bounds__(NW * 32, kCtasPerSm<QMODE, NG, PAIR>)
    paged_decode_quant_balanced_kernel(QDecodeArgs a, int batch, int nwt_launch) {
    constexpr int KSTEPS = D / 16;
    constexpr int MT = D / 16;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, c = lane & 3;
    // the merge grid may be scheduled now; it waits for this grid to finish
    asm volatile("griddepcontrol.launch_dependents;");
    __shared__ uint4 sq[NW][PAIR ? 2 : 1][KSTEPS / 2][32];
    __shared__ __align__(16) float sm_o[NW][8][D];

    const int i = blockIdx.x * NW + warp;
    WarpSplit sp;
    bool bad = false;
    const bool any =
        sp.begin(a.ctx_lens, batch, a.max_blocks * BS, a.hkv, nwt_launch, kBalancedMinItems, i, bad);
    if (i == 0 && bad && lane == 0) atomicOr(a.status, PKV_STATUS_BAD_CONTEXT);
    if (!any) return;
    while (sp.next()) {
        QState<MT, NG> st;
        quant_pass<T, D, QMODE, NG, WIN, PAIR>(a, sp.b, sp.kvh, sp.ctx, sp.lb0, sp.lb1, 1, &sq[warp][0][0][lane],
                                               st);
        quant_finish<D, QMODE, NG>(st);
        // partial (m, l, o) of this run: o staged through shared memory so
        // the G x D rows go out in 16-byte stores
        __syncwarp();
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            int dl, dh;
            out_columns<D, QMODE, NG>(mt, g, dl, dh);
            sm_o[warp][2 * c][dl] = st.o[mt][0];
            sm_o[warp][2 * c + 1][dl] = st.o[mt][1];
            sm_o[warp][2 * c][dh] = st.o[mt][2];
            sm_o[warp][2 * c + 1][dh] = st.o[mt][3];
        }
        __syncwarp();
        const int64_t slot = i + static_cast<int64_t>(sp.b) * a.hkv + sp.kvh;
        float4* po = reinterpret_cast<float4*>(a.ws_o + slot * a.G * D);
        const float4* so = reinterpret_cast<const float4*>(&sm_o[warp][0][0]);
        for (int x = lane; x < a.G * D / 4; x += 32) po[x] = so[x];
        if (g == 0) {
            float* pml = a.ws_ml + slot * a.G * 2;
            if (2 * c < a.G) {
                pml[4 * c] = st.m0;
                pml[4 * c + 1] = st.l0;
            }
            if (2 * c + 1 < a.G) {
                pml[4 * c + 2] = st.m1;
                pml[4 * c + 3] = st.l1;
            }
        }
    }
}

// Whether a call takes the paired-block pass (INT4 with at most 4 query
// heads per KV head: two blocks fit the MMA's 8 query columns).
inline bool use_pairs(int qmode, int G) { return qmode == PKV_QMODE_INT4_ASYM && G <= 4; }

template <typename T, int D, int QMODE, int NG, bool PAIR>
void launch_balanced_w(const QDecodeArgs& a, int batch, int nwt, cudaStream_t st) {
    const dim3 grid((nwt + NW - 1) / NW);
    if (a.window > 0)
        paged_decode_quant_balanced_kernel<T, D, QMODE, NG, true, PAIR><<<grid, NW * 32, 0, st>>>(a, batch, nwt);
    else
        paged_decode_quant_balanced_kernel<T, D, QMODE, NG, false, PAIR><<<grid, NW * 32, 0, st>>>(a, batch, nwt);
}

template <typename T, int D, int QMODE, int NG>
void launch_balanced(const QDecodeArgs& a, int batch, int nwt, cudaStream_t st) {
    if constexpr (QMODE == PKV_QMODE_INT4_ASYM) {
        if (use_pairs(QMODE, a.G)) return launch_balanced_w<T, D, QMODE, NG, true>(a, batch, nwt, st);
    }
    launch_balanced_w<T, D, QMODE, NG, false>(a, batch, nwt, st);
}

template <typename T, int D, int QMODE, int NG, bool SPLIT, bool PAIR>
void launch_w(const QDecodeArgs& a, int parts, int hkv, int batch, cudaStream_t st) {
    dim3 grid(SPLIT ? parts : 1, hkv, batch);
    if (a.window > 0) paged_decode_quant_kernel<T, D, QMODE, NG, true, SPLIT, PAIR><<<grid, NW * 32, 0, st>>>(a);
    else paged_decode_quant_kernel<T, D, QMODE, NG, false, SPLIT, PAIR><<<grid, NW * 32, 0, st>>>(a);
}

template <typename T, int D, int QMODE, int NG, bool SPLIT>
void launch(const QDecodeArgs& a, int parts, int hkv, int batch, cudaStream_t st) {
    if constexpr (QMODE == PKV_QMODE_INT4_ASYM) {
        if (use_pairs(QMODE, a.G)) return launch_w<T, D, QMODE, NG, SPLIT, true>(a, parts, hkv, batch, st);
    }
    launch_w<T, D, QMODE, NG, SPLIT, false>(a, parts, hkv, batch, st);
}

// The kernel for (dtype, head dim, mode, column groups); balanced or
// partitioned (SPLIT: partials, else a single pass).
template <bool BALANCED, bool SPLIT>
int dispatch(const QDecodeArgs& a, int D, int qmode, int ng, int dtype, int parts, int hkv, int batch,
             int nwt, cudaStream_t st) {
#define PKV_Q(TT, DD, QM, NN)                                                          \
    do {                                                                                 \
        if (BALANCED) launch_balanced<TT, DD, QM, NN>(a, batch, nwt, st);              \
        else launch<TT, DD, QM, NN, SPLIT>(a, parts, hkv, batch, st);                   \
    } while (0)
#define PKV_QT(TT)                                                                       \
    do {                                                                                 \
        if (qmode == PKV_QMODE_INT4_ASYM) {                                              \
            if (D == 128 && ng == 2) PKV_Q(TT, 128, PKV_QMODE_INT4_ASYM, 2);             \
            else if (D == 128) PKV_Q(TT, 128, PKV_QMODE_INT4_ASYM, 1);                   \
            else PKV_Q(TT, 64, PKV_QMODE_INT4_ASYM, 1);                                  \
        } else {                                                                         \
            if (D == 128) PKV_Q(TT, 128, PKV_QMODE_FP8_E4M3, 1);                         \
            else PKV_Q(TT, 64, PKV_QMODE_FP8_E4M3, 1);                                   \
        }                                                                                \
    } while (0)
    if (dtype == PKV_DTYPE_BF16) PKV_QT(__nv_bfloat16);
    else PKV_QT(__half);
#undef PKV_QT
#undef PKV_Q
    return launch_status();
}

}  // namespace
}  // namespace pkv

extern "C" int pkv_paged_attention_decode_quant(
    const void* q, const void* k_codes, const void* k_scale, const void* k_zero, const void* v_codes,
    const void* v_scale, const void* v_zero, const void* sink_k, const void* sink_v, int32_t n_sink,
    const void* win_k, const void* win_v, int32_t window, const int32_t* block_tables, const int32_t* context_lens, int32_t batch, int32_t num_q_heads,
    int32_t num_kv_heads, int32_t head_dim, int32_t num_blocks, int32_t block_size,
    int32_t max_blocks, int32_t group_size, float scale, void* out, void* workspace,
    size_t workspace_bytes, int32_t partition_size, int qmode, int dtype, void* stream) {
    if (batch < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || num_blocks <= 0 ||
        block_size <= 0 || max_blocks < 0 || partition_size < 0 || n_sink < 0 || window < 0)
        return PKV_ERR_INVALID_ARG;
    if (dtype != PKV_DTYPE_F16 && dtype != PKV_DTYPE_BF16) return PKV_ERR_INVALID_ARG;
    if (qmode != PKV_QMODE_INT4_ASYM && qmode != PKV_QMODE_FP8_E4M3) return PKV_ERR_INVALID_ARG;
    if (num_q_heads % num_kv_heads != 0) return PKV_ERR_INVALID_ARG;
    if (block_size != pkv::BS || (head_dim != 64 && head_dim != 128) ||
        num_q_heads / num_kv_heads > 8 || n_sink > pkv::BS || batch > 65535 || num_kv_heads > 65535)
        return PKV_ERR_UNSUPPORTED;
    // INT4 groups: one per (token, head), or 64 columns at head dim 128
    const int ng = qmode == PKV_QMODE_INT4_ASYM && group_size > 0 ? head_dim / group_size : 1;
    if (qmode == PKV_QMODE_INT4_ASYM &&
        !(group_size == head_dim || (head_dim == 128 && group_size == 64)))
        return PKV_ERR_UNSUPPORTED;
    const int32_t ps = partition_size == 0
                           ? pkv::auto_partition_size(batch, num_q_heads, static_cast<int64_t>(max_blocks) * pkv::BS)
                           : partition_size;
    if (ps % block_size != 0) return PKV_ERR_INVALID_ARG;
    if (batch == 0) return PKV_OK;
    if (!q || !k_codes || !k_scale || !v_codes || !v_scale || !block_tables || !context_lens || !out)
        return PKV_ERR_INVALID_ARG;
    if (qmode == PKV_QMODE_INT4_ASYM && (!k_zero || !v_zero)) return PKV_ERR_INVALID_ARG;
    if (n_sink > 0 && (!sink_k || !sink_v)) return PKV_ERR_INVALID_ARG;
    if (window % block_size != 0) return PKV_ERR_INVALID_ARG;
    if (window > 0 && (!win_k || !win_v)) return PKV_ERR_INVALID_ARG;
    if (window > 0 && (!pkv::aligned16(win_k) || !pkv::aligned16(win_v))) return PKV_ERR_MISALIGNED;
    if (!pkv::aligned16(q) || !pkv::aligned16(k_codes) || !pkv::aligned16(v_codes) ||
        !pkv::aligned16(out) || (reinterpret_cast<uintptr_t>(k_scale) & 1u) ||
        (reinterpret_cast<uintptr_t>(v_scale) & 1u))
        return PKV_ERR_MISALIGNED;
    int* st = pkv::status_word();
    if (!st) return PKV_ERR_CUDA;
    pkv::QDecodeArgs a;
    a.q = q;
    a.k_codes = static_cast<const uint8_t*>(k_codes);
    a.k_scale = static_cast<const __half*>(k_scale);
    a.k_zero = static_cast<const __half*>(k_zero);
    a.v_codes = static_cast<const uint8_t*>(v_codes);
    a.v_scale = static_cast<const __half*>(v_scale);
    a.v_zero = static_cast<const __half*>(v_zero);
    a.sink_k = sink_k;
    a.sink_v = sink_v;
    a.n_sink = n_sink;
    a.win_k = win_k;
    a.win_v = win_v;
    a.window = window;
    a.ring = window / block_size + 1;
    a.tables = block_tables;
    a.ctx_lens = context_lens;
    a.hq = num_q_heads;
    a.hkv = num_kv_heads;
    a.G = num_q_heads / num_kv_heads;
    a.num_blocks = num_blocks;
    a.max_blocks = max_blocks;
    a.part_blocks = ps / block_size;
    a.max_parts = (max_blocks + a.part_blocks - 1) / a.part_blocks;
    if (a.max_parts < 1) a.max_parts = 1;
    a.scale_log2 = scale * pkv::kLog2e;
    a.out = out;
    a.ws_o = nullptr;
    a.ws_ml = nullptr;
    a.status = st;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    if (partition_size == 0 && a.max_parts > 1 && pkv::use_balanced(batch, num_kv_heads, max_blocks)) {
        // balanced split, all CTAs resident: kCtasPerSm CTAs of NW warps per SM
        const int per_sm =
            pkv::NW * (qmode != PKV_QMODE_INT4_ASYM ? pkv::kCtasPerSm<PKV_QMODE_FP8_E4M3>
                       : pkv::use_pairs(qmode, a.G) ? pkv::kCtasPerSm<PKV_QMODE_INT4_ASYM, 1, true>
                       : ng == 2                    ? pkv::kCtasPerSm<PKV_QMODE_INT4_ASYM, 2>
                                                    : pkv::kCtasPerSm<PKV_QMODE_INT4_ASYM, 1>);
        const int nwt = pkv::balanced_warps(static_cast<int64_t>(batch) * num_kv_heads * max_blocks, per_sm);
        const size_t rows = static_cast<size_t>(nwt) * a.G + static_cast<size_t>(batch) * num_q_heads;
        if (!workspace || workspace_bytes < pkv::balanced_bytes(batch, num_q_heads, a.G, head_dim, nwt))
            return PKV_ERR_WORKSPACE;
        if (!pkv::aligned16(workspace)) return PKV_ERR_MISALIGNED;
        a.ws_o = static_cast<float*>(workspace);
        a.ws_ml = a.ws_o + rows * head_dim;
        int r = pkv::dispatch<true, true>(a, head_dim, qmode, ng, dtype, 0, num_kv_heads, batch, nwt, cs);
        if (r != PKV_OK) return r;
        return pkv::launch_balanced_merge(context_lens, batch, num_q_heads, num_kv_heads, head_dim,
                                          max_blocks * block_size, nwt, a.ws_o, a.ws_ml, out, dtype, cs);
    }
    if (a.max_parts <= 1) {
        a.part_blocks = max_blocks > 0 ? max_blocks : 1;
        return pkv::dispatch<false, false>(a, head_dim, qmode, ng, dtype, 1, num_kv_heads, batch, 0, cs);
    }
    const size_t need = static_cast<size_t>(batch) * num_q_heads * a.max_parts * (head_dim + 2) * sizeof(float);
    if (!workspace || workspace_bytes < need) return PKV_ERR_WORKSPACE;
    if (!pkv::aligned16(workspace)) return PKV_ERR_MISALIGNED;
    a.ws_o = static_cast<float*>(workspace);
    a.ws_ml = a.ws_o + static_cast<size_t>(batch) * num_q_heads * a.max_parts * head_dim;
    int r = pkv::dispatch<false, true>(a, head_dim, qmode, ng, dtype, a.max_parts, num_kv_heads, batch, 0, cs);
    if (r != PKV_OK) return r;
    return pkv_paged_attention_decode_merge(context_lens, batch, num_q_heads, head_dim, max_blocks,
                                            block_size, ps, workspace, workspace_bytes, out, dtype,
                                            stream);
}
