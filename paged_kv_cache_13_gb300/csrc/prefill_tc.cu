// Multi-query paged attention over long query spans (chunked-prefill slices)
// on the 5th-generation tensor cores: tcgen05.mma with the accumulators in
// tensor memory (TMEM), K/V tiles gathered from the paged pool by TMA.
//
// What it computes: exactly pkv_paged_attention_multi_query (multi_query.cu):
// query token i of sequence b sits at position p = ctx_b - L_b + i and
//   out[q_start[b] + i, h] = sum_{t <= p} softmax_t(scale <q, K_t>) V_t
// over KV head h / G ("The 8GB VRAM Breakthrough", §5 "Chunked Prefill": a
// 512-token slice of a prompt attends to the cache before it and causally
// to itself).
//
// Design (one CTA of 12 warps per 128 query rows of one (sequence, KV head);
// a row is a (query token, query head) pair, 128 / G tokens per tile):
// * Q tile [128 rows x 128 dims] bf16/fp16 in shared memory; K and V tiles
//   of 128 keys (8 pool blocks) in 2-stage rings, each block's 16 rows
//   fetched by one TMA box straight from its physical block (unused or bad
//   blocks become rows past the map's end, which TMA fills with zeros).
// * Warps 0-7 (two warpgroups, 232 registers each after setmaxnreg) do the
//   softmax; warps 8-11 (one warpgroup, 40 registers) issue: lane 0 of warp
//   8 the S MMAs, lane 0 of warp 9 the O MMAs, warps 10 and 11 the K and V
//   copies (a lane per block, the table entries loaded by the same lanes
//   two tiles ahead).  An MMA issue blocks while the tensor pipe drains (16
//   MMAs of a tile take ~1,200 cycles to issue), so no softmax warp issues
//   any.
// * S = Q K^T (M 128, N 128, K 128: 8 tcgen05.mma of K 16) into one of two
//   TMEM S buffers (columns [0, 128) and [256, 384)): S(j + 1) is computed
//   while the softmax of tile j runs.  Softmax warps w and w + 4 share the
//   TMEM lanes (rows) 32 (w % 4) .. +31, each taking 64 of the 128 columns:
//   the thread of row r loads its half row of S, applies the causal mask
//   (only on tiles that reach past the CTA's first query position), and the
//   two halves exchange their maxima through shared memory under a barrier
//   of just those two warps, for the online softmax (base 2, the reference
//   max raised only by more than 8).
// * P (bf16: P and its rounding residual, two operands, so the products see
//   ~16 bits of P) is written into TMEM over its own S buffer, and O += P V
//   (M 128, N 128, K 128 keys) takes A from TMEM, B (V) from shared memory,
//   into TMEM columns [128, 256); S(j + 2) is issued once O += P(j) V(j) has
//   read the buffer.  A rescale of O (when a row's reference max moves) is
//   a TMEM load / store of that half row.  O / l goes out at the end.
// * Hand-offs are mbarriers: K / V landed (TMA), S done and O done
//   (tcgen05.commit), P written (one arrival per softmax warp), the V stage
//   and P buffer read (a second commit).  Each waiter is at most one phase
//   behind its barrier by construction (a barrier's next phase needs the
//   waiter's own later arrival).
// * Every shared-memory operand tile is a grid of 8-row x 128-byte swizzle
//   atoms (128-byte swizzle).  In Q atom (g, h) -- rows 8g .. 8g+7, columns
//   64h .. 64h+63 -- sits at byte h * 16 KiB + g * 1 KiB of the tile; in K
//   and V (one TMA box per 16-row block, so its two row groups and two
//   column halves land together) at g * 2 KiB + h * 1 KiB.  K-major
//   operands (Q, K) step 32 bytes per K-16 slice inside an atom row; V is
//   the MN-major B operand of O += P V (its 8-key groups 2 KiB apart, its
//   two 64-dim halves 1 KiB apart).
// * Every wait suspends in hardware (try_wait) and is bounded in time: one
//   that runs out sets PKV_STATUS_COPY_TIMEOUT and the stop flag; softmax
//   warp pairs stop together (the OR their barrier returns), the issuers
//   let their MMAs and copies in flight finish (bounded), and the CTA still
//   frees its TMEM.

#include <cuda.h>

#include <mutex>
#include <type_traits>

#include "balanced.cuh"
#include "prefill_tc.cuh"

namespace pkv {
namespace {

constexpr int kRows = 128;   // query rows per CTA (MMA M)
constexpr int kKeys = 128;   // keys per tile (MMA N of S, K of O)
constexpr int kDim = 128;    // head dim
constexpr int kBS = 16;      // tokens per pool block
constexpr int kTile = kRows * kDim * 2;  // bytes of one 128 x 128 16-bit tile
// warps 0-7: softmax, two per 32-row TMEM lane quarter; warps 8-11: producers
constexpr int kSoftmaxWarps = 8;
constexpr int kWarpS = 8;   // lane 0 issues S = Q K^T
constexpr int kWarpO = 9;   // lane 0 issues O += P V
constexpr int kWarpK = 10;  // K copies
constexpr int kWarpV = 11;  // V copies
constexpr int kThreads = 384;
// Registers: launched at 168 a thread (384 threads, one CTA per SM), the
// softmax warpgroups raise theirs to 232 and the producer warpgroup lowers
// its own to 40 (setmaxnreg): 2 x 128 x 232 + 128 x 40 = 384 x 168.
constexpr int kLaunchRegs = 168;
constexpr int kNoBlock = -2147483647 - 1;  // a tile slot past the context

// Test hook (pkv_debug_prefill_drop_copy): the K copy of this key tile is
// never issued (-1: off), so the S issuer's bounded wait for it runs out.
__device__ int g_drop_copy_tile = -1;
static_assert(2 * 128 * 232 + 128 * 40 <= kThreads * kLaunchRegs, "register split exceeds the launch's registers");
constexpr int kTmemCols = 512;  // the whole TMEM: one CTA per SM (shared memory)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kSlack = 8.f;
// time after which an mbarrier wait gives up (ns): a wait that will never
// complete ends within ~0.3 s
constexpr uint64_t kWaitNs = 300000000ull;

// shared-memory map (bytes from the 1 KiB-aligned base)
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kTile;      // 2 stages
constexpr int kOffV = kOffK + 2 * kTile;  // 2 stages
constexpr int kOffBar = kOffV + 2 * kTile;           // mbarriers, then the TMEM address and stop flag
constexpr int kOffXch = kOffBar + 256;                // [2][128] floats: row values of the two halves
// mbarriers (index: count)
constexpr int kBarKFull = 0;   // 2 (per stage): the K tile has landed (TMA)
constexpr int kBarVFull = 2;   // 2: the V tile has landed
constexpr int kBarSFull = 4;   // 2 (per S buffer): S = Q K^T done
constexpr int kBarO = 6;       // O += P V done: O may be touched
constexpr int kBarP = 7;       // 8 (softmax warps): P written into TMEM, O rescaled
constexpr int kBarVFree = 8;   // 2 (per stage / buffer): O += P V done reading V and P
constexpr int kNumBars = 10;
constexpr int kSmemBytes = kOffXch + 2 * 128 * 4 + 1024;  // then alignment slack

struct TcArgs {
    const void* q;
    const int32_t* q_start;
    const int32_t* tables;
    const int32_t* ctx_lens;
    int hq, hkv, G, num_blocks, max_blocks, total_rows;
    float scale_log2;
    void* out;
    int* status;
};

// ---------------------------------------------------------------- PTX
__device__ __forceinline__ uint32_t sh_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// one plain arrival
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// one arrival that also expects `bytes` of copies to complete on the barrier
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Waits for the barrier's phase of the given parity; false if it has not
// completed within kWaitNs.  try_wait suspends the thread in hardware until
// the phase completes or a short system time limit passes, so a waiting
// warp takes no issue slots from the warps still working.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity) {
    uint64_t t0 = 0;
    for (int it = 0;; ++it) {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(bar), "r"(parity)
            : "memory");
        if (done) return true;
        if (it == 0) t0 = global_ns();
        else if (global_ns() - t0 > kWaitNs) return false;
    }
}

// One 16-row block of the pool (4 KiB) as a 4-D box: coordinates (0, 0, 0,
// w), w the block's first 8-row group (see pool_map).
__device__ __forceinline__ void tma_load_block(uint32_t dst, const CUtensorMap* map, int w, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %2, %2, "
        "%3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(w), "r"(bar)
        : "memory");
}

// UMMA shared-memory descriptor: start, leading and stride byte offsets (16-
// byte units), version 1, 128-byte swizzle.
__device__ __forceinline__ uint64_t smem_desc(uint32_t start, uint32_t lbo, uint32_t sbo) {
    return static_cast<uint64_t>((start >> 4) & 0x3FFFu) | (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
           (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor of kind::f16: fp32 accumulator, A and B of the
// 16-bit type (bf16 or fp16), K-major A, B K-major or MN-major, M 128, N 128.
template <typename T>
__device__ __forceinline__ uint32_t instr_desc(bool b_mn_major) {
    constexpr uint32_t fmt = std::is_same<T, __nv_bfloat16>::value ? 1u : 0u;
    return (1u << 4) | (fmt << 7) | (fmt << 10) | (static_cast<uint32_t>(b_mn_major) << 16) |
           (static_cast<uint32_t>(kKeys >> 3) << 17) | (static_cast<uint32_t>(kRows >> 4) << 24);
}

__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, bool acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(static_cast<uint32_t>(acc))
        : "memory");
}

// the same with A read from TMEM (lane = row, K elements packed two per
// 32-bit column), B from shared memory
__device__ __forceinline__ void mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc, bool acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b), "r"(idesc), "r"(static_cast<uint32_t>(acc))
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void fence_before_sync() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after_sync() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 32 consecutive TMEM columns of this thread's lane (warp w: lanes 32w ..)
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
        "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
        "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
    uint32_t r[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(v[i]);
    tmem_st32(taddr, r);
}

// max of three floats (one instruction on sm_100 and later)
__device__ __forceinline__ float max3f(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// named barrier of the 64 threads of softmax warps w and w + 4 (id 1 .. 4)
__device__ __forceinline__ void pair_sync(int id) {
    asm volatile("bar.sync %0, 64;" ::"r"(id) : "memory");
}

// the same barrier, returning whether any of the 64 threads passed true
__device__ __forceinline__ bool pair_sync_or(int id, bool pred) {
    uint32_t any;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %2, 0;\n\t"
        "bar.red.or.pred q, %1, 64, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(any)
        : "r"(id), "r"(static_cast<uint32_t>(pred))
        : "memory");
    return any != 0;
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Byte offset of element (row r, column col) in a swizzled 128 x 128 tile.
__device__ __forceinline__ uint32_t tile_off(int r, int col) {
    return (col >> 6) * 16384 + (r >> 3) * 1024 + (r & 7) * 128 + ((((col & 63) >> 3) ^ (r & 7)) << 4) +
           (col & 7) * 2;
}

template <typename T>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    return Half16<T>::pack(lo, hi);
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap, TcArgs a) {
    constexpr bool kSplit = std::is_same<T, __nv_bfloat16>::value;
    constexpr int kHalf = kKeys / 2;  // columns of S (and O) per softmax thread
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = sh_addr(sm);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kOffBar);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kOffBar + 112);
    int* abort_flag = reinterpret_cast<int*>(sm + kOffBar + 116);
    float* xch = reinterpret_cast<float*>(sm + kOffXch);  // [2][128]: per-half row values
    const uint32_t bar0 = sh_addr(bars);
    auto bar = [&](int i) { return bar0 + 8 * i; };

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool softmax = warp < kSoftmaxWarps;
    // softmax warp w: TMEM lanes (rows) 32 (w % 4) .. +31, columns 64 (w / 4) .. +63
    const int r = 32 * (warp & 3) + lane, hc = (warp >> 2) & 1;
    const int tile = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
    const int q0 = a.q_start[b], L = a.q_start[b + 1] - q0;
    const int tpt = kRows / a.G;  // query tokens per tile
    const int tok0 = tile * tpt;
    if (L <= 0 || tok0 >= L) return;
    int ctx = a.ctx_lens[b];
    const int cap = a.max_blocks * kBS;
    if (ctx < L || ctx > cap) {
        if (tid == 0 && tile == 0 && kvh == 0) atomicOr(a.status, PKV_STATUS_BAD_CONTEXT);
        ctx = ctx > cap ? cap : ctx;
    }
    const int first_pos = ctx - L;
    const int last_tok = min(tok0 + tpt, L) - 1;
    const int last_pos = first_pos + last_tok;  // the tile's last query position
    const int ntiles = last_pos >= 0 ? last_pos / kKeys + 1 : 0;
    const int nblk = (ctx + kBS - 1) / kBS;  // blocks holding context tokens

    if (tid == 0) {
        for (int i = 0; i < kNumBars; ++i)
            mbar_init(bar(i), i == kBarP ? kSoftmaxWarps : 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(sh_addr(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }

    // ---- Q tile: softmax thread (r, hc) writes columns 64 hc .. +63 of row r
    const int my_tok = tok0 + r / a.G, my_h = r - (r / a.G) * a.G;
    if (softmax) {
        const bool valid = my_tok < L;
        const uint4* src = valid ? reinterpret_cast<const uint4*>(
                                       static_cast<const T*>(a.q) +
                                       ((static_cast<int64_t>(q0) + my_tok) * a.hq + kvh * a.G + my_h) * kDim) +
                                       hc * 8
                                 : nullptr;
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
            const uint4 v = valid ? src[ch] : make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4*>(sm + kOffQ + tile_off(r, hc * 64 + ch * 8)) = v;
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // Q visible to the MMA
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tO = tmem + kKeys;  // S buffers at columns 0 and 256, O at 128
    auto tS = [&](int s) { return tmem + (s ? 2 * kKeys : 0); };
    const int32_t* trow = a.tables + static_cast<int64_t>(b) * a.max_blocks;
    auto stopped = [&]() { return *reinterpret_cast<volatile int*>(abort_flag) != 0; };
    auto give_up = [&]() {
        atomicOr(a.status, PKV_STATUS_COPY_TIMEOUT);
        *reinterpret_cast<volatile int*>(abort_flag) = 1;
    };

    if (!softmax) {
        // ================= producers: S issuer, O issuer, K copies, V copies
        asm volatile("setmaxnreg.dec.sync.aligned.u32 40;");
        if (warp == kWarpS && lane == 0) {
            // S(j) = Q K(j)^T into S buffer j % 2, once K(j) has landed and
            // O += P(j - 2) V(j - 2) has read P(j - 2) out of that buffer
            const uint32_t idesc = instr_desc<T>(false);
            int last = -1;
            for (int j = 0; j < ntiles && !stopped(); ++j) {
                const int s = j & 1;
                if (!wait_bar(bar(kBarKFull + s), (j >> 1) & 1) ||
                    (j >= 2 && !wait_bar(bar(kBarVFree + s), ((j - 2) >> 1) & 1))) {
                    give_up();
                    break;
                }
                fence_after_sync();
                const uint32_t qa = sbase + kOffQ, kb = sbase + kOffK + s * kTile;
#pragma unroll
                for (int kk = 0; kk < kDim / 16; ++kk) {
                    // Q: halves at 16 KiB, 8-row groups at 1 KiB; K: halves
                    // at 1 KiB, 8-key groups at 2 KiB
                    const uint32_t qoff = (kk >> 2) * 16384 + (kk & 3) * 32, koff = (kk >> 2) * 1024 + (kk & 3) * 32;
                    mma_f16(tS(s), smem_desc(qa + qoff, 16384, 1024), smem_desc(kb + koff, 1024, 2048), idesc,
                            kk > 0);
                }
                mma_commit(bar(kBarSFull + s));
                last = j;
            }
            // stopping early: let the S MMAs in flight finish (bounded)
            if (stopped() && last >= 0) wait_bar(bar(kBarSFull + (last & 1)), (last >> 1) & 1);
        } else if (warp == kWarpO && lane == 0) {
            // O += P(j) V(j), once the softmax has written P(j) and V(j) has
            // landed; its completion frees P, O and V stage j % 2
            const uint32_t idesc = instr_desc<T>(true);
            int last = -1;
            for (int j = 0; j < ntiles && !stopped(); ++j) {
                const int s = j & 1;
                if (!wait_bar(bar(kBarP), j & 1) || !wait_bar(bar(kBarVFull + s), (j >> 1) & 1)) {
                    give_up();
                    break;
                }
                fence_after_sync();
                const uint32_t vb = sbase + kOffV + s * kTile;
#pragma unroll
                for (int kk = 0; kk < kKeys / 16; ++kk) {
                    // P of keys 16 kk .. +15: TMEM columns 8 kk .. +7 of S
                    // buffer s (its residual 64 columns further); V of block
                    // kk: halves (N) at 1 KiB, 8-key groups (K) at 2 KiB
                    const uint64_t bd = smem_desc(vb + kk * 4096, 1024, 2048);
                    mma_f16_ts(tO, tS(s) + kk * 8, bd, idesc, j > 0 || kk > 0);
                    if constexpr (kSplit) mma_f16_ts(tO, tS(s) + kKeys / 2 + kk * 8, bd, idesc, true);
                }
                mma_commit(bar(kBarO));
                mma_commit(bar(kBarVFree + s));
                last = j;
            }
            if (stopped() && last >= 0) wait_bar(bar(kBarO), last & 1);
        } else if (warp == kWarpK || warp == kWarpV) {
            // TMA copies of tile t into stage t % 2, one 16-row block per lane
            // (lanes 0-7); stage t % 2 is free for K once S(t - 2) is done,
            // for V once O(t - 2) is done.  The table entries are loaded two
            // tiles before their copies, so the warp never waits on those
            // loads.  (Prefetching the rows into L2 ahead of the copies, one
            // bulk prefetch per block, cost more than it saved once the copy
            // engine was the busiest unit: 368 -> 340 us without it.)
            const bool is_v = warp == kWarpV;
            const int jj = lane & 7;
            const bool copier = lane < 8;
            const int drop = is_v ? -1 : *reinterpret_cast<volatile int*>(&g_drop_copy_tile);
            const uint32_t base = sbase + (is_v ? kOffV : kOffK);
            const CUtensorMap* map = is_v ? &vmap : &kmap;
            // the physical block of block jj of tile t (kNoBlock: none), and its TMA
            // row: the load is only consumed a tile or two later, and nothing
            // branches on it before then (a bad id is reported once, at the end)
            auto entry_at = [&](int t) {
                const int lb = t * 8 + jj;
                return t < ntiles && lb < nblk ? __ldg(trow + lb) : kNoBlock;
            };
            bool bad = false;
            auto row_of = [&](int phys) {
                const bool ok = static_cast<unsigned>(phys) < static_cast<unsigned>(a.num_blocks);
                bad |= phys != kNoBlock && !ok;
                return ok ? (phys * a.hkv + kvh) * kBS : a.total_rows;
            };
            // entries of tiles t and t + 1
            int e = copier ? entry_at(0) : kNoBlock;
            int e_next = copier ? entry_at(1) : kNoBlock;
            int issued = 0;
            for (int t = 0; t < ntiles; ++t) {
                const int s = t & 1;
                const int e_after = copier ? entry_at(t + 2) : kNoBlock;
                const int y = row_of(e);
                int go = 1;
                if (lane == 0) {
                    go = !stopped();
                    if (go && t >= 2) {
                        go = is_v ? wait_bar(bar(kBarVFree + s), ((t - 2) >> 1) & 1)
                                  : wait_bar(bar(kBarSFull + s), ((t - 2) >> 1) & 1);
                        if (!go) give_up();
                    }
                }
                if (!__shfl_sync(0xffffffffu, go, 0)) break;
                if (copier && t != drop) {
                    const uint32_t fb = bar((is_v ? kBarVFull : kBarKFull) + s);
                    if (lane == 0) mbar_arrive_expect_tx(fb, kTile);
                    tma_load_block(base + s * kTile + jj * 4096, map, y >> 3, fb);
                }
                e = e_next;
                e_next = e_after;
                issued = t + 1;
            }
            if (bad && !is_v) atomicOr(a.status, PKV_STATUS_BAD_BLOCK);
            // stopping early: let the copies in flight land (bounded) before
            // the shared memory is given up
            if (lane == 0 && stopped()) {
                for (int t = issued - 1; t >= 0 && t >= issued - 2; --t)
                    wait_bar(bar((is_v ? kBarVFull : kBarKFull) + (t & 1)), (t >> 1) & 1);
            }
            __syncwarp();
        }
    } else {
        // ================= softmax warps
        asm volatile("setmaxnreg.inc.sync.aligned.u32 232;");
        const int my_pos = my_tok < L ? first_pos + my_tok : -1;  // padding rows: all masked
        const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
        float m = neg_inf(), l = 0.f;  // l: this thread's half of the row sum
        bool late = false;  // a wait after the pair exchange ran out: stop at the next one
        for (int j = 0; j < ntiles; ++j) {
            const int s = j & 1;
            // ---- this thread's half row of S(j), masked and scaled (base 2)
            const bool want = !late && !__any_sync(0xffffffffu, stopped());
            const bool have_s = want && __all_sync(0xffffffffu, wait_bar(bar(kBarSFull + s), (j >> 1) & 1));
            float x[kHalf];
            if (have_s) {
                fence_after_sync();
#pragma unroll
                for (int cc = 0; cc < kHalf / 32; ++cc) {
                    float v[32];
                    tmem_ld32(tS(s) + lane_base + hc * kHalf + cc * 32, v);
#pragma unroll
                    for (int i = 0; i < 32; ++i) x[cc * 32 + i] = v[i];
                }
                tmem_wait_ld();
            } else {
#pragma unroll
                for (int i = 0; i < kHalf; ++i) x[i] = neg_inf();
            }
            // A tile wholly at or below the CTA's first query position needs
            // no causal mask (padding rows there see zero queries: finite
            // scores, outputs never written).  With a positive scale the max
            // is taken over raw scores and the scale enters the exponent's
            // FMA (mul); otherwise the scores are scaled first.
            const int key0 = j * kKeys + hc * kHalf;
            const bool interior = j * kKeys + kKeys - 1 <= first_pos + tok0;
            const float mul = a.scale_log2 > 0.f ? a.scale_log2 : 1.f;
            if (a.scale_log2 > 0.f) {
                if (!interior) {
#pragma unroll
                    for (int i = 0; i < kHalf; ++i)
                        if (key0 + i > my_pos) x[i] = neg_inf();
                }
            } else {
#pragma unroll
                for (int i = 0; i < kHalf; ++i) x[i] = key0 + i <= my_pos ? x[i] * a.scale_log2 : neg_inf();
            }
            // the half row's max: three-input max, four independent chains
            float mq[4] = {x[0], x[1], x[2], x[3]};
#pragma unroll
            for (int i = 4; i < kHalf; i += 8) {
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    mq[u] = max3f(mq[u], x[i + u], x[i + 4 + u < kHalf ? i + 4 + u : i + u]);
            }
            float mx = max3f(mq[0], mq[1], fmaxf(mq[2], mq[3])) * mul;
            // the row max over both halves; warps w and w + 4 (the two halves
            // of the same rows) meet here and stop together if either lacks S
            xch[hc * kRows + r] = mx;
            if (pair_sync_or(1 + (warp & 3), !have_s)) break;
            mx = fmaxf(mx, xch[(1 - hc) * kRows + r]);
            const bool raise = mx > m + kSlack;
            float alpha = 1.f;
            if (raise) {
                alpha = m == neg_inf() ? 0.f : ex2(m - mx);
                m = mx;
                l *= alpha;
            }
            // P of this half row, packed (bf16: value and rounding residual),
            // written over S(j) in TMEM: the thread's row (lane), keys
            // 64 hc .. +63 as 32 columns from column 32 hc of the buffer,
            // their residuals 64 columns further (the partner warp has read
            // its half of S(j): it passed the pair barrier).  P of the
            // previous tile sits in the other buffer; the store still waits
            // for the previous O += P V, which has mostly finished while the
            // exponentials ran: without that wait three of four runs of the
            // parity tests had one CTA's row wrong (cause not found).
            const float mref = m == neg_inf() ? 0.f : m;
            float sum = 0.f;
            uint32_t phi[kHalf / 2], plo[kSplit ? kHalf / 2 : 1];
#pragma unroll
            for (int i = 0; i < kHalf; i += 2) {
                const float p0 = ex2(fmaf(x[i], mul, -mref)), p1 = ex2(fmaf(x[i + 1], mul, -mref));
                sum += p0 + p1;
                phi[i / 2] = pack2<T>(p0, p1);
                if constexpr (kSplit)
                    plo[i / 2] = pack2<T>(p0 - __uint_as_float(phi[i / 2] << 16),
                                          p1 - __uint_as_float(phi[i / 2] & 0xffff0000u));
            }
            l += sum;
            if (j > 0 && !__all_sync(0xffffffffu, wait_bar(bar(kBarO), (j - 1) & 1))) {
                if (lane == 0) give_up();
                late = true;
                continue;
            }
            fence_after_sync();
            tmem_st32(tS(s) + lane_base + hc * (kHalf / 2), phi);
            if constexpr (kSplit) tmem_st32(tS(s) + lane_base + kKeys / 2 + hc * (kHalf / 2), plo);
            // a moved reference max: O is rescaled before this tile's P V
            // adds to it
            if (j > 0 && __any_sync(0xffffffffu, raise)) {
#pragma unroll
                for (int cc = 0; cc < kHalf / 32; ++cc) {
                    float v[32];
                    tmem_ld32(tO + lane_base + hc * kHalf + cc * 32, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] *= alpha;
                    tmem_st32(tO + lane_base + hc * kHalf + cc * 32, v);
                }
            }
            tmem_wait_st();
            // keys past the context in this tile: their V rows may hold any
            // bits (0 x NaN would poison O); zero them once the tile has landed
            if (j * kKeys + kKeys > ctx) {
                if (!__all_sync(0xffffffffu, wait_bar(bar(kBarVFull + s), (j >> 1) & 1))) {
                    if (lane == 0) give_up();
                    late = true;
                    continue;
                }
                if (j * kKeys + r >= ctx) {
                    uint4* row = reinterpret_cast<uint4*>(sm + kOffV + s * kTile + (r >> 4) * 4096 +
                                                          ((r >> 3) & 1) * 2048 + hc * 1024 + (r & 7) * 128);
#pragma unroll
                    for (int ch = 0; ch < 8; ++ch) row[ch] = make_uint4(0, 0, 0, 0);
                }
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // zeroed V rows to the MMA
            fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(kBarP));  // P(j) written, O rescaled
        }
        // the row sum over both halves
        xch[hc * kRows + r] = l;
        pair_sync(1 + (warp & 3));
        l += xch[(1 - hc) * kRows + r];

        // ---- epilogue: O / l for this thread's half row
        bool ok = !stopped() && ntiles > 0;
        if (ok && !wait_bar(bar(kBarO), (ntiles - 1) & 1)) {
            atomicOr(a.status, PKV_STATUS_COPY_TIMEOUT);
            ok = false;
        }
        fence_after_sync();
        T* orow = static_cast<T*>(a.out) + ((static_cast<int64_t>(q0) + my_tok) * a.hq + kvh * a.G + my_h) * kDim;
        if (__any_sync(0xffffffffu, ok)) {  // warp-collective TMEM loads
            const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
            for (int cc = 0; cc < kHalf / 32; ++cc) {
                float v[32];
                tmem_ld32(tO + lane_base + hc * kHalf + cc * 32, v);
                tmem_wait_ld();
                if (ok && my_tok < L) {
                    uint4* dst = reinterpret_cast<uint4*>(orow + hc * kHalf + cc * 32);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        uint4 w;
                        w.x = pack2<T>(v[8 * q] * inv, v[8 * q + 1] * inv);
                        w.y = pack2<T>(v[8 * q + 2] * inv, v[8 * q + 3] * inv);
                        w.z = pack2<T>(v[8 * q + 4] * inv, v[8 * q + 5] * inv);
                        w.w = pack2<T>(v[8 * q + 6] * inv, v[8 * q + 7] * inv);
                        dst[q] = w;
                    }
                }
            }
        } else if (ntiles == 0 && my_tok < L) {  // every position negative: zeros
            for (int d = hc * kHalf; d < hc * kHalf + kHalf; ++d) orow[d] = Half16<T>::from_float(0.f);
        }
    }
    fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        fence_after_sync();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols)
                     : "memory");
    }
}

// ---------------------------------------------------------------- host
using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encode_fn() {
    static std::once_flag once;
    static EncodeTiled fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiled>(p);
    });
    return fn;
}

// The pool [num_blocks * Hkv * 16 rows, 128 dims] as a 4-D tensor: (64
// dims; 8 rows at 256 bytes; 2 column halves at 128 bytes; 8-row groups at
// 2 KiB).  A box (64, 8, 2, 2) is one 16-row block, 4 KiB, landing as
// [group][half][row][64 dims] with 128-byte swizzle: one copy per block
// where a 2-D map takes two (one per 128-byte column half), and the copy
// engine's cost is mostly per copy (measured on GB300: a 32 KiB tile of 8
// blocks takes ~1,450 cycles as 8 such boxes, ~1,790 as 16 2-D boxes).
bool pool_map(CUtensorMap* map, const void* pool, int64_t rows, bool bf16) {
    EncodeTiled enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[4] = {64, 8, 2, static_cast<cuuint64_t>(rows / 8)};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(kDim) * 2, 128, static_cast<cuuint64_t>(kDim) * 2 * 8};
    const cuuint32_t box[4] = {64, 8, 2, 2};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return enc(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4,
               const_cast<void*>(pool), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename T>
int launch_t(const CUtensorMap& km, const CUtensorMap& vm, const TcArgs& a, int tiles, int batch, cudaStream_t st) {
    static std::once_flag once;
    static cudaError_t attr = cudaSuccess;
    static int regs = 0;
    std::call_once(once, [] {
        attr = cudaFuncSetAttribute(prefill_tc_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        cudaFuncAttributes fa;
        if (attr == cudaSuccess && (attr = cudaFuncGetAttributes(&fa, prefill_tc_kernel<T>)) == cudaSuccess)
            regs = fa.numRegs;
    });
    if (attr != cudaSuccess) return PKV_ERR_CUDA;
    // the warpgroups' register split needs the launch's full allocation
    if (regs < kLaunchRegs) return PKV_ERR_UNSUPPORTED;
    prefill_tc_kernel<T><<<dim3(tiles, a.hkv, batch), kThreads, kSmemBytes, st>>>(km, vm, a);
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace

bool prefill_tc_applies(int head_dim, int G, int64_t rows) {
    return head_dim == kDim && (G == 1 || G == 2 || G == 4 || G == 8) && rows > kPrefillTcMinRows;
}

int launch_prefill_tc(const void* q, const int32_t* q_start, const void* k_pool, const void* v_pool,
                      const int32_t* tables, const int32_t* ctx_lens, int batch, int hq, int hkv, int num_blocks,
                      int max_blocks, int max_q_len, float scale, void* out, int* status, bool bf16,
                      cudaStream_t st) {
    const int64_t rows = static_cast<int64_t>(num_blocks) * hkv * kBS;
    if (rows >= (1LL << 31)) return PKV_ERR_UNSUPPORTED;
    CUtensorMap km, vm;
    if (!pool_map(&km, k_pool, rows, bf16) || !pool_map(&vm, v_pool, rows, bf16)) return PKV_ERR_CUDA;
    TcArgs a;
    a.q = q;
    a.q_start = q_start;
    a.tables = tables;
    a.ctx_lens = ctx_lens;
    a.hq = hq;
    a.hkv = hkv;
    a.G = hq / hkv;
    a.num_blocks = num_blocks;
    a.max_blocks = max_blocks;
    a.total_rows = static_cast<int>(rows);
    a.scale_log2 = scale * kLog2e;
    a.out = out;
    a.status = status;
    const int tpt = kRows / a.G;
    const int tiles = (max_q_len + tpt - 1) / tpt;
    return bf16 ? launch_t<__nv_bfloat16>(km, vm, a, tiles, batch, st) : launch_t<__half>(km, vm, a, tiles, batch, st);
}

}  // namespace pkv

extern "C" int pkv_debug_prefill_drop_copy(int32_t tile) {
    if (tile < -1) return PKV_ERR_INVALID_ARG;
    return cudaMemcpyToSymbol(pkv::g_drop_copy_tile, &tile, sizeof(tile)) == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}
