// backward_tc.cuh -- gradients of the Lizard operator on tcgen05 tensor cores
// (bf16 inputs, d = 128, window w <= 65), chunk-parallel.
//
// Operator (Lizard, gist.science/de section 2 items 1-3): gated linear
// attention S_t = diag(sigmoid(g_t)) S_{t-1} + k_t^T v_t, yg_t = q_t S_t, an
// anchor window with meta-memory sinks, and y = yg + alpha ya.  The backward
// is split at chunk boundaries (C = 64 tokens, b = in-chunk base-2 prefix of
// log sigmoid(g), the log-space form of the page's "Hardware-bewusster
// Algorithmus"):
//
//   chunk_states_kernel  one CTA per (unit, direction) walks the chunks once:
//       forward:  Sb[c] = state before chunk c,
//                 S <- diag(2^{b_last}) S + (k 2^{b_last - b})^T v
//       reverse:  Ha[c] = dLoss/d(state after chunk c),
//                 H <- diag(2^{b_last}) H + (q 2^{b})^T dy
//   bwd_query_kernel     one CTA per (unit, chunk): the window softmax of the
//       chunk's rows (log-normaliser, D_t = alpha dy_t . ya_t, taken as
//       alpha sum_s P_ts (dy v^T)_ts with P in fp32), dq, and
//       q * dq_gate for dg, d mu and d alpha
//   bwd_key_kernel       one CTA per (unit, chunk): dk and dv (gate terms
//       from Ha[c], the anchor terms of this chunk's and the next chunk's
//       rows), and dg from the reverse prefix of q dq - k dk, whose later
//       chunks' share sum_j S_after[i][j] Ha[c][i][j] is regrouped (see E2)
//       so that nothing cancels but fp32 rounding.
// States and state gradients are kept in bf16, row = key dim.
//
// Head dim d = 64 (template DH) runs on the same 128-wide tiles: the dims
// 64..127 of every input tile are cleared at the CTA's start and the TMA
// loads only the first 64-dim box, so every product and state sees zeros
// there; the scratch (states, q * dq_gate) keeps the 128-wide layout, and
// only dims < d of dq, dk, dv, dg, d meta_k are written.
#pragma once

#include <type_traits>

#include "common.cuh"
#include "prefill_ws.cuh"
#include "sm100.cuh"

namespace lizard {
namespace bwdtc {

using namespace sm100;
using ws::bf2_to_f2;
using ws::ex2;
using ws::f2_to_bf2;
using ws::log2_sigmoid;
using ws::LOG2E;
using ws::tlane;

constexpr int C = 64;
constexpr int D = 128;
constexpr int THREADS = 256;
constexpr uint32_t TILE = C * 128;  // one 64-row x 128-byte swizzled block (8 KB)
constexpr uint32_t WAIT = 1u << 21;

// A 16-byte global load issued where it is written: volatile, so the
// compiler keeps it ahead of the waits that follow instead of sinking it to
// its first use (a prefetch meant to overlap them).
__device__ __forceinline__ uint4 ldg_early(const void *p)
{
    uint4 r;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// Clears the 64-dim blocks past the head dim of a CTA's input tiles (d = 64:
// the TMA then loads only the first block of each).  `blk` lists the byte
// offsets of those blocks (8 KB each, rows of 128 B).
template <int N>
__device__ __forceinline__ void clear_blocks(uint8_t *sm, const uint32_t (&blk)[N], uint32_t bytes)
{
    for (uint32_t e = threadIdx.x; e < N * (bytes / 16); e += blockDim.x)
        *reinterpret_cast<uint4 *>(sm + blk[e / (bytes / 16)] + 16 * (e % (bytes / 16))) = make_uint4(0u, 0u, 0u, 0u);
}

// Bounded wait on an mbarrier phase by every thread of the CTA; false (and
// the device error word set) on timeout.
__device__ __forceinline__ bool cta_wait(uint64_t *bar, uint32_t phase)
{
    const bool ok = mbar_wait(bar, phase & 1u, WAIT);
    if (!ok) atomicExch(&g_device_error, DEV_TIMEOUT);
    return __syncthreads_and(ok) != 0;
}

// In-chunk base-2 prefix sums of log sigmoid(g) for key dims 2p, 2p+1 and
// tokens 16 hq .. 16 hq + 15 (rows >= n: no decay), from a swizzled g tile.
// Returns b for the thread's 16 tokens; fills tot[4][128] (quarter totals)
// and needs one __syncthreads before `finish_prefix`.
struct Prefix {
    float2 b[16];
};
__device__ __forceinline__ void local_prefix(const uint8_t *gtile, int p, int hq, int n, Prefix &pf, float *tot)
{
    const uint32_t kblk = (p / 32) * TILE, kbyte = (p % 32) * 4;
    float2 run = make_float2(0.f, 0.f);
#pragma unroll
    for (int tt = 0; tt < 16; ++tt) {
        const int t = 16 * hq + tt;
        const float2 g = bf2_to_f2(*reinterpret_cast<const uint32_t *>(gtile + kblk + sw128_offset(t, kbyte)));
        if (t < n) {
            run.x += log2_sigmoid(g.x);
            run.y += log2_sigmoid(g.y);
        }
        pf.b[tt] = run;
    }
    tot[hq * 128 + 2 * p] = run.x;
    tot[hq * 128 + 2 * p + 1] = run.y;
}
// The same from gate logits held in registers (bf16 pairs of dims 2p, 2p+1).
__device__ __forceinline__ void local_prefix_regs(const uint32_t (&gr)[16], int p, int hq, int n, Prefix &pf,
                                                  float *tot)
{
    float2 run = make_float2(0.f, 0.f);
#pragma unroll
    for (int tt = 0; tt < 16; ++tt) {
        const float2 g = bf2_to_f2(gr[tt]);
        if (16 * hq + tt < n) {
            run.x += log2_sigmoid(g.x);
            run.y += log2_sigmoid(g.y);
        }
        pf.b[tt] = run;
    }
    tot[hq * 128 + 2 * p] = run.x;
    tot[hq * 128 + 2 * p + 1] = run.y;
}
// Adds the earlier quarters' totals; returns b_last (the chunk total).
__device__ __forceinline__ float2 finish_prefix(int p, int hq, Prefix &pf, const float *tot)
{
    float2 off = make_float2(0.f, 0.f), all = make_float2(0.f, 0.f);
#pragma unroll
    for (int qq = 0; qq < 4; ++qq) {
        const float2 t2 = make_float2(tot[qq * 128 + 2 * p], tot[qq * 128 + 2 * p + 1]);
        if (qq < hq) {
            off.x += t2.x;
            off.y += t2.y;
        }
        all.x += t2.x;
        all.y += t2.y;
    }
#pragma unroll
    for (int tt = 0; tt < 16; ++tt) {
        pf.b[tt].x += off.x;
        pf.b[tt].y += off.y;
    }
    return all;
}

// ============================================================ chunk states
struct StatesArgs {
    __nv_bfloat16 *Sb;       // [units][nchunks][D][D]  state before chunk c
    __nv_bfloat16 *Ha;       // [units][nchunks][D][D]  dLoss/d(state after chunk c)
    const __nv_bfloat16 *g;  // [units][L][D] gate logits (read into registers a chunk ahead)
    int L, nchunks;
    int H, group;            // query heads per key/value head (tk, tv map B x H / group heads)
};

// Shared memory (about 100 KB, two CTAs per SM): two stages of (x, y)
// tiles, two operand tiles, vectors.
constexpr uint32_t ST_STAGE = 2 * 2 * TILE;                 // x | y, 16 KB each
constexpr uint32_t ST_OP = 2 * ST_STAGE;                    // operand tiles [2] (16 KB each)
constexpr uint32_t ST_VEC = ST_OP + 2 * 2 * TILE;           // dec[128], tot[4][128]
constexpr uint32_t ST_BAR = ST_VEC + (128 + 512) * 4;       // bars: tma[2], mma
constexpr uint32_t ST_TSLOT = ST_BAR + 3 * 8;
constexpr uint32_t ST_SMEM = ST_TSLOT + 8 + 1024;

// grid (units, 2): blockIdx.y = 0 walks forward (maps x = k, y = v), 1 walks
// backward (x = q, y = dy).  Per chunk, with X the walked matrix kept
// transposed in tensor memory (lane = value dim j, column = key dim i):
//   store X (row i = key dim) to out[c]; X^T <- X^T diag(2^{b_last}) + y^T O,
//   O = k 2^{b_last - b} (forward) or q 2^{b} (backward).
template <int DH>
__global__ void __launch_bounds__(THREADS, 2)
    chunk_states_kernel(const __grid_constant__ CUtensorMap tg, const __grid_constant__ CUtensorMap tk,
                        const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tq,
                        const __grid_constant__ CUtensorMap tdy, const StatesArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = smem_align1024(smem_raw);
    const uint32_t sb = smem_u32(sm);
    float *dec = reinterpret_cast<float *>(sm + ST_VEC), *tot = dec + 128;
    uint64_t *bar_tma = reinterpret_cast<uint64_t *>(sm + ST_BAR), *bar_mma = bar_tma + 2;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + ST_TSLOT);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int unit = blockIdx.x;
    const bool rev = blockIdx.y == 1;
    const int L = a.L, nch = a.nchunks;
    const CUtensorMap *mx = rev ? &tq : &tk, *my = rev ? &tdy : &tv;
    __nv_bfloat16 *out = (rev ? a.Ha : a.Sb) + (size_t)unit * nch * D * D;
    constexpr int d = DH, nbox = DH / 64;
    if constexpr (DH < D) {
        const uint32_t blk[4] = {TILE, 3 * TILE, ST_STAGE + TILE, ST_STAGE + 3 * TILE};  // x, y block 1 of both stages
        clear_blocks(sm, blk, TILE);
        fence_proxy_async_smem();
    }

    if (warp == 0) {
        tmem_alloc(tslot, 128);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(&bar_tma[0], 1);
        mbar_init(&bar_tma[1], 1);
        mbar_init(bar_mma, 1);
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    if (warp < 4) {  // X = 0
        uint32_t z[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) z[e] = 0u;
        for (int cc = 0; cc < D; cc += 16) tmem_st16(tmem + tlane(warp) + cc, z);
        tmem_wait_st();
    }
    auto chunk_of = [&](int idx) { return rev ? nch - 1 - idx : idx; };
    const int xyu = rev ? unit : kv_unit(unit, a.H, a.group);  // k, v come from the key/value head
    auto issue = [&](int idx) {
        const int c = chunk_of(idx), s = idx & 1;
        uint8_t *st = sm + s * ST_STAGE;
        mbar_arrive_expect_tx(&bar_tma[s], 2 * nbox * TILE);
        for (int x = 0; x < nbox; ++x) {
            tma_load_3d(st + x * TILE, mx, &bar_tma[s], 64 * x, c * C, xyu);
            tma_load_3d(st + (2 + x) * TILE, my, &bar_tma[s], 64 * x, c * C, xyu);
        }
    };
    if (tid == 0) issue(0);
    uint32_t tma_use[2] = {0, 0}, mma_use = 0, mma_issued = 0, tma_issued[2] = {1, 0};
    bool ok = true;
    const int p = tid & 63, hq = tid >> 6;
    const uint32_t id_st = instr_desc(128, 128, FMT_BF16, 1, 1);
    // gate logits of dims 2p, 2p+1 for this thread's 16 tokens, one chunk ahead
    // (dims past d read as g = 0: their x and y are zero)
    const uint32_t *gp = reinterpret_cast<const uint32_t *>(a.g + (size_t)unit * L * d) + p;
    uint32_t gnext[16];
    auto load_g = [&](int idx) {
        const int c = chunk_of(idx);
#pragma unroll
        for (int tt = 0; tt < 16; ++tt) {
            const int row = c * C + 16 * hq + tt;
            gnext[tt] = row < L && 2 * p < d ? gp[(size_t)row * (d / 2)] : 0u;
        }
    };
    load_g(0);

    for (int idx = 0; idx < nch && ok; ++idx) {
        const int c = chunk_of(idx), s = idx & 1;
        const int n = min(C, L - c * C);
        uint8_t *st = sm + s * ST_STAGE;
        uint32_t gcur[16];
#pragma unroll
        for (int tt = 0; tt < 16; ++tt) gcur[tt] = gnext[tt];
        if (idx + 1 < nch) load_g(idx + 1);
        ok = cta_wait(&bar_tma[s], tma_use[s]);
        if (!ok) break;
        ++tma_use[s];
        // gate prefix and the operand tile O[s]
        Prefix pf;
        local_prefix_regs(gcur, p, hq, n, pf, tot);
        __syncthreads();
        const float2 bl = finish_prefix(p, hq, pf, tot);
        if (hq == 0) {
            dec[2 * p] = ex2(bl.x);
            dec[2 * p + 1] = ex2(bl.y);
        }
        {
            const uint32_t kblk = (p / 32) * TILE, kbyte = (p % 32) * 4;
            uint8_t *op = sm + ST_OP + s * 2 * TILE;
#pragma unroll
            for (int tt = 0; tt < 16; ++tt) {
                const int t = 16 * hq + tt;
                const uint32_t o = kblk + sw128_offset(t, kbyte);
                const float2 x = bf2_to_f2(*reinterpret_cast<const uint32_t *>(st + o));
                const float2 e = rev ? make_float2(ex2(pf.b[tt].x), ex2(pf.b[tt].y))
                                     : make_float2(ex2(bl.x - pf.b[tt].x), ex2(bl.y - pf.b[tt].y));
                *reinterpret_cast<uint32_t *>(op + o) = f2_to_bf2(x.x * e.x, x.y * e.y);
            }
        }
        fence_proxy_async_smem();
        // the previous chunk's product is done: stage s^1 and O[s^1] are free
        if (idx >= 1) {
            ok = cta_wait(bar_mma, mma_use);
            if (!ok) break;
            ++mma_use;
        }
        if (tid == 0 && idx + 1 < nch) {
            issue(idx + 1);
            ++tma_issued[(idx + 1) & 1];
        }
        tc_fence_after();
        {
            // store X (this chunk's entry), then decay it: warp w takes
            // lanes 32 (w % 4) .. + 31 and columns 64 (w / 4) .. + 63
            const int q4 = warp & 3, ch = warp >> 2;
            const int j = 32 * q4 + lane;
            __nv_bfloat16 *o = out + (size_t)c * D * D + j;
#pragma unroll 1
            for (int cc = 64 * ch; cc < 64 * ch + 64; cc += 32) {
                uint32_t r0[16], r1[16];
                tmem_ld16(tmem + tlane(q4) + cc, r0);
                tmem_ld16(tmem + tlane(q4) + cc + 16, r1);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const float x0 = __uint_as_float(r0[e]), x1 = __uint_as_float(r1[e]);
                    o[(size_t)(cc + e) * D] = __float2bfloat16_rn(x0);
                    o[(size_t)(cc + 16 + e) * D] = __float2bfloat16_rn(x1);
                    r0[e] = __float_as_uint(x0 * dec[cc + e]);
                    r1[e] = __float_as_uint(x1 * dec[cc + 16 + e]);
                }
                tmem_st16(tmem + tlane(q4) + cc, r0);
                tmem_st16(tmem + tlane(q4) + cc + 16, r1);
            }
            tmem_wait_st();
        }
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (tid == 0) {
            const uint32_t yb = sb + s * ST_STAGE + 2 * TILE, ob = sb + ST_OP + s * 2 * TILE;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_bf16_ss(tmem, smem_desc(yb + kk * 2048, TILE, 1024), smem_desc(ob + kk * 2048, TILE, 1024),
                            id_st, 1u);
            mma_commit(bar_mma);
            ++mma_issued;
        }
    }
    // Drain: every product and copy issued has completed before shared and
    // tensor memory are released (bounded).
    if (tid == 0) {
        for (uint32_t i = mma_use; i < mma_issued; ++i)
            if (!mbar_wait(bar_mma, i & 1u, WAIT)) break;
        for (int s2 = 0; s2 < 2; ++s2)
            for (uint32_t i = tma_use[s2]; i < tma_issued[s2]; ++i)
                if (!mbar_wait(&bar_tma[s2], i & 1u, WAIT)) break;
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 128);
}

// ============================================================ query side
struct QueryArgs {
    const __nv_bfloat16 *mu, *k;  // meta keys [H][m][D]; keys (for the exact path)
    __nv_bfloat16 *dq;            // [units][L][D]
    float *xq;                    // [units][L][D]  q * dq_gate
    float *lse2, *drow;           // [units][L]     base-2 log-normaliser, D_t
    float *dmu;                   // [H][m][D]      accumulated (zeroed by the host)
    float *dalpha;                // accumulated (zeroed by the host): [H] with alpha_h, else one value
    float alpha;
    int H, L, w, m, nchunks;
    const float *alpha_h;         // per-head anchor weights (null: alpha)
    int group;                    // query heads per key/value head
};

constexpr int META_ROWS = 16;
constexpr uint32_t KB_K = (C + META_ROWS) * 128;  // one 64-dim block of the current key tile (80 rows)
constexpr float SPAN2_MAX = 100.f;                 // half-chunk decay span limit (base 2) of the folded operands
// Shared memory of bwd_query_kernel (offsets from a 1024-aligned base).
constexpr uint32_t QO_Q = 0;                    // q      [64][128]  (2 blocks)
constexpr uint32_t QO_DY = QO_Q + 2 * TILE;     // dy
constexpr uint32_t QO_G = QO_DY + 2 * TILE;     // g
constexpr uint32_t QO_KP = QO_G + 2 * TILE;     // k of the previous chunk
constexpr uint32_t QO_KC = QO_KP + 2 * TILE;    // k of this chunk + meta keys (80 rows, 2 blocks of KB_K)
constexpr uint32_t QO_V = QO_KC + 2 * KB_K;     // v prev | v cur (4 blocks); later the state (128 x 128)
constexpr uint32_t QO_KR = QO_V + 4 * TILE;     // k 2^{r - b}
constexpr uint32_t QO_DA = QO_KR + 2 * TILE;    // tril(dy v^T) of this chunk [64][64]
constexpr uint32_t QO_DSC = QO_DA + TILE;       // score gradients [64][prev 64 | cur 64 | meta 16]
constexpr uint32_t QO_B = QO_DSC + 3 * TILE;    // b fp32 [64][128]
constexpr uint32_t QO_VEC = QO_B + C * D * 4;   // r[128], tot[4][128], dC[64][16], flags
constexpr uint32_t QO_BAR = QO_VEC + (128 + 512 + 64 * 16 + 4) * 4;
constexpr uint32_t QO_TSLOT = QO_BAR + 4 * 8;
constexpr uint32_t QO_SMEM = QO_TSLOT + 8 + 1024;
static_assert(QO_SMEM <= 232448, "shared memory budget");
// Tensor-memory columns (512): window scores, dy v^T; later the three parts
// of dq.
constexpr uint32_t QT_SC = 0, QT_DP = 144;
constexpr uint32_t QT_G1 = 0, QT_G2 = 128, QT_DQA = 256;

// grid = units * nchunks: CTA (unit, chunk c).
template <int DH>
__global__ void __launch_bounds__(THREADS, 1)
    bwd_query_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                     const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tg,
                     const __grid_constant__ CUtensorMap tdy, const __grid_constant__ CUtensorMap tS,
                     const QueryArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = smem_align1024(smem_raw);
    const uint32_t sb = smem_u32(sm);
    float *rv = reinterpret_cast<float *>(sm + QO_VEC), *tot = rv + 128, *dC = tot + 512;
    int *flags = reinterpret_cast<int *>(dC + 64 * 16);
    float *bq = reinterpret_cast<float *>(sm + QO_B);
    // Element (t, i) of bq sits at column i ^ (t mod 32) of row t: a warp
    // reading one column of 16 rows (two column halves) hits 32 banks.
    auto bx = [](int t, int i) { return t * D + (i ^ (t & 31)); };
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + QO_BAR);
    uint64_t *bar_in = bars, *bar_s = bars + 1, *bar_mma = bars + 2;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + QO_TSLOT);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nch = a.nchunks;
    const int unit = blockIdx.x / nch, c = blockIdx.x % nch, h = unit % a.H;
    const int L = a.L, w = a.w, m = a.m;
    const int c0 = c * C, n = min(C, L - c0);
    const bool has_prev = c > 0;
    const float alpha = head_alpha(a.alpha_h, a.alpha, h);
    const int kvu = kv_unit(unit, a.H, a.group);

    if (warp == 0) {
        tmem_alloc(tslot, 512);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int i = 0; i < 3; ++i) mbar_init(&bars[i], 1);
        flags[0] = 0;
        fence_mbar_init();
    }
    constexpr int d = DH, nbox = DH / 64;
    if constexpr (DH < D) {
        // block 1 of q, dy, g, the keys (their 64 token rows), the values
        const uint32_t blk[7] = {QO_Q + TILE, QO_DY + TILE, QO_G + TILE, QO_KP + TILE, QO_KC + KB_K, QO_V + TILE,
                                 QO_V + 3 * TILE};
        clear_blocks(sm, blk, TILE);
    }
    // meta keys into rows 64..79 of the current key tile (zero past m and d)
    for (int e = tid; e < META_ROWS * 64; e += THREADS) {
        const int r = e / 64, ip = e % 64, i = 2 * ip;
        uint32_t val = 0u;
        if (r < m && i < d) val = *reinterpret_cast<const uint32_t *>(a.mu + ((size_t)h * m + r) * d + i);
        *reinterpret_cast<uint32_t *>(sm + QO_KC + (i / 64) * KB_K + sw128_offset(C + r, (i % 64) * 2)) = val;
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    uint32_t mma_use = 0, mma_issued = 0, in_issued = 0, s_issued = 0;

    if (tid == 0) {
        const uint32_t bytes = (has_prev ? 7 : 5) * nbox * TILE;
        mbar_arrive_expect_tx(bar_in, bytes);
        for (int hb = 0; hb < nbox; ++hb) {
            tma_load_3d(sm + QO_Q + hb * TILE, &tq, bar_in, 64 * hb, c0, unit);
            tma_load_3d(sm + QO_DY + hb * TILE, &tdy, bar_in, 64 * hb, c0, unit);
            tma_load_3d(sm + QO_G + hb * TILE, &tg, bar_in, 64 * hb, c0, unit);
            tma_load_3d(sm + QO_KC + hb * KB_K, &tk, bar_in, 64 * hb, c0, kvu);
            tma_load_3d(sm + QO_V + (2 + hb) * TILE, &tv, bar_in, 64 * hb, c0, kvu);
            if (has_prev) {
                tma_load_3d(sm + QO_KP + hb * TILE, &tk, bar_in, 64 * hb, c0 - C, kvu);
                tma_load_3d(sm + QO_V + hb * TILE, &tv, bar_in, 64 * hb, c0 - C, kvu);
            }
        }
        in_issued = 1;
    }
    auto mma_wait = [&]() -> bool {
        const bool r = cta_wait(bar_mma, mma_use);
        if (r) ++mma_use;
        return r;
    };
    int unsafe = 0;
    do {
        if (!cta_wait(bar_in, 0)) break;
        // ---- prep: b (base-2 in-chunk prefix), r = b at token 31, KR = k 2^{r - b}
        {
            const int p = tid & 63, hq = tid >> 6;
            Prefix pf;
            local_prefix(sm + QO_G, p, hq, n, pf, tot);
            __syncthreads();
            finish_prefix(p, hq, pf, tot);
            if (hq == 1) {
                rv[2 * p] = pf.b[15].x;
                rv[2 * p + 1] = pf.b[15].y;
            }
            __syncthreads();
            const float2 r2 = make_float2(rv[2 * p], rv[2 * p + 1]);
            const uint32_t kblk = (p / 32) * TILE, kbyte = (p % 32) * 4;
            bool wide = false;
#pragma unroll
            for (int tt = 0; tt < 16; ++tt) {
                const int t = 16 * hq + tt;
                const float2 bt = pf.b[tt];
                wide |= fabsf(bt.x - r2.x) > SPAN2_MAX || fabsf(bt.y - r2.y) > SPAN2_MAX;
                bq[bx(t, 2 * p)] = bt.x;
                bq[bx(t, 2 * p + 1)] = bt.y;
                const float2 kv = bf2_to_f2(*reinterpret_cast<const uint32_t *>(
                    sm + QO_KC + (p / 32) * KB_K + sw128_offset(t, kbyte)));
                *reinterpret_cast<uint32_t *>(sm + QO_KR + kblk + sw128_offset(t, kbyte)) =
                    f2_to_bf2(kv.x * ex2(r2.x - bt.x), kv.y * ex2(r2.y - bt.y));
            }
            unsafe = __syncthreads_or(wide);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        // ---- M1: window + meta scores, dy v^T over the band
        if (tid == 0) {
            const uint32_t id64 = instr_desc(64, 64, FMT_BF16, 0, 0), id80 = instr_desc(64, 80, FMT_BF16, 0, 0);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint32_t ko = (kk / 4) * TILE + (kk % 4) * 32;
                const uint64_t qd = smem_desc(sb + QO_Q + ko, 16, 1024), dyd = smem_desc(sb + QO_DY + ko, 16, 1024);
                if (has_prev) {
                    mma_bf16_ss(tmem + QT_SC, qd, smem_desc(sb + QO_KP + ko, 16, 1024), id64, kk > 0);
                    mma_bf16_ss(tmem + QT_DP, dyd, smem_desc(sb + QO_V + ko, 16, 1024), id64, kk > 0);
                }
                mma_bf16_ss(tmem + QT_SC + 64, qd, smem_desc(sb + QO_KC + (kk / 4) * KB_K + (kk % 4) * 32, 16, 1024),
                            id80, kk > 0);
                mma_bf16_ss(tmem + QT_DP + 64, dyd, smem_desc(sb + QO_V + 2 * TILE + ko, 16, 1024), id64, kk > 0);
            }
            mma_commit(bar_mma);
            ++mma_issued;
        }
        if (!mma_wait()) break;
        // the value tiles are read (by dy v^T): load this chunk's state into their place
        if (tid == 0) {
            mbar_arrive_expect_tx(bar_s, 4 * TILE);  // four 64 x 64 boxes
            const int z = unit * nch + c;
            for (int jb = 0; jb < 2; ++jb)
                for (int ib = 0; ib < 2; ++ib)
                    tma_load_3d(sm + QO_V + jb * 2 * TILE + ib * TILE, &tS, bar_s, 64 * jb, 64 * ib, z);
            s_issued = 1;
        }
        tc_fence_after();
        // ---- E1: row softmax (warps 0-3, row t, column half hs), tril(dA) (warps 4-7)
        const int quarter = warp & 3, hs = lane >> 4;
        const int t = 16 * quarter + (lane & 15);
        const uint32_t tl = tmem + tlane(quarter);
        const int hi = t + 64, lo = max(has_prev ? 0 : 64, hi - w + 1);  // band columns of row t
        const bool rowok = t < n;
        float lse2 = 0.f;
        if (warp < 4) {
            uint32_t r[4][16], rm[16];
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) tmem_ld16_x2<16>(tl + QT_SC + 32 * jj, r[jj]);
            tmem_ld16(tl + QT_SC + 128, rm);
            tmem_wait_ld();
            float mx = -INFINITY;
#pragma unroll
            for (int jj = 0; jj < 4; ++jj)
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int col = 32 * jj + 16 * hs + e;
                    if (col >= lo && col <= hi) mx = fmaxf(mx, __uint_as_float(r[jj][e]));
                }
#pragma unroll
            for (int e = 0; e < META_ROWS; ++e)
                if (hs == 0 && e < m) mx = fmaxf(mx, __uint_as_float(rm[e]));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
            const float M2 = mx * LOG2E;
            float sum = 0.f;
#pragma unroll
            for (int jj = 0; jj < 4; ++jj)
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int col = 32 * jj + 16 * hs + e;
                    if (col >= lo && col <= hi) sum += ex2(fmaf(__uint_as_float(r[jj][e]), LOG2E, -M2));
                }
#pragma unroll
            for (int e = 0; e < META_ROWS; ++e)
                if (hs == 0 && e < m) sum += ex2(fmaf(__uint_as_float(rm[e]), LOG2E, -M2));
            sum += __shfl_xor_sync(0xffffffffu, sum, 16);
            lse2 = M2 + ws::lg2(sum);
            if (rowok && hs == 0) a.lse2[(size_t)unit * L + c0 + t] = lse2;
            if (hs == 0) tot[t] = lse2;  // for warps 4-7 (tot is free after the prep)
        } else {
            uint32_t r[2][16];
            tmem_ld16_x2<16>(tl + QT_DP + 64, r[0]);
            tmem_ld16_x2<16>(tl + QT_DP + 96, r[1]);
            tmem_wait_ld();
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
                const int s0 = 32 * jj + 16 * hs;
                uint32_t pk[8];
#pragma unroll
                for (int e = 0; e < 16; e += 2)
                    pk[e / 2] = f2_to_bf2((rowok && s0 + e <= t) ? __uint_as_float(r[jj][e]) : 0.f,
                                          (rowok && s0 + e + 1 <= t) ? __uint_as_float(r[jj][e + 1]) : 0.f);
                *reinterpret_cast<uint4 *>(sm + QO_DA + sw128_offset(t, s0 * 2)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                *reinterpret_cast<uint4 *>(sm + QO_DA + sw128_offset(t, s0 * 2 + 16)) =
                    make_uint4(pk[4], pk[5], pk[6], pk[7]);
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        tc_fence_after();
        // ---- E2: D_t = alpha dy . ya, d alpha; score gradients; d mu.
        // D_t = alpha sum_j dy_tj sum_s P_ts v_sj = alpha sum_s P_ts dP_ts
        // with dP = dy v^T (the sinks carry no value): P in fp32, recomputed
        // from the scores and the row's log-normaliser.
        // All eight warps: warp w takes rows 16 (w % 4) .. + 15 and the
        // column groups jj = 2 (w / 4), 2 (w / 4) + 1 (32 columns each).
        {
            const int g = warp >> 2;
            if (g == 1) lse2 = tot[t];
            uint32_t rd[2][16];
            float pr[2][16];
            {
                uint32_t r[2][16];
#pragma unroll
                for (int jx = 0; jx < 2; ++jx) {
                    tmem_ld16_x2<16>(tl + QT_SC + 32 * (2 * g + jx), r[jx]);
                    tmem_ld16_x2<16>(tl + QT_DP + 32 * (2 * g + jx), rd[jx]);
                }
                tmem_wait_ld();
#pragma unroll
                for (int jx = 0; jx < 2; ++jx)
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int col = 32 * (2 * g + jx) + 16 * hs + e;
                        const bool valid = rowok && col >= lo && col <= hi;
                        pr[jx][e] = valid ? ex2(fmaf(__uint_as_float(r[jx][e]), LOG2E, -lse2)) : 0.f;
                    }
            }
            float dot = 0.f;
#pragma unroll
            for (int jx = 0; jx < 2; ++jx)
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    dot = pr[jx][e] != 0.f ? fmaf(pr[jx][e], __uint_as_float(rd[jx][e]), dot) : dot;
            dot += __shfl_xor_sync(0xffffffffu, dot, 16);
            float *part = tot + 128;  // [2][64] row partials of the two column halves
            if (hs == 0) part[64 * g + t] = dot;
            __syncthreads();
            dot = part[t] + part[64 + t];
            if (!rowok) dot = 0.f;
            const float Dt = alpha * dot;
            if (g == 0) {
                if (rowok && hs == 0) a.drow[(size_t)unit * L + c0 + t] = Dt;
                // d alpha: this warp's rows
                float da = hs == 0 ? dot : 0.f;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) da += __shfl_xor_sync(0xffffffffu, da, o);
                if (lane == 0) atomicAdd(a.dalpha + (a.alpha_h ? h : 0), da);
            }
            // dSC = P (alpha dP - D_t) over the band, dC = P_meta (0 - D_t)
#pragma unroll
            for (int jx = 0; jx < 2; ++jx) {
                const int col0 = 32 * (2 * g + jx) + 16 * hs;
                uint32_t pk[8];
#pragma unroll
                for (int e = 0; e < 16; e += 2) {
                    float dv2[2];
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int col = col0 + e + u;
                        const bool valid = rowok && col >= lo && col <= hi;
                        dv2[u] = valid ? pr[jx][e + u] * (alpha * __uint_as_float(rd[jx][e + u]) - Dt) : 0.f;
                    }
                    pk[e / 2] = f2_to_bf2(dv2[0], dv2[1]);
                }
                const uint32_t o = QO_DSC + (col0 / 64) * TILE;
                *reinterpret_cast<uint4 *>(sm + o + sw128_offset(t, (col0 % 64) * 2)) =
                    make_uint4(pk[0], pk[1], pk[2], pk[3]);
                *reinterpret_cast<uint4 *>(sm + o + sw128_offset(t, (col0 % 64) * 2 + 16)) =
                    make_uint4(pk[4], pk[5], pk[6], pk[7]);
            }
            if (g == 1) {
                uint32_t rm[16];
                tmem_ld16(tl + QT_SC + 128, rm);
                tmem_wait_ld();
                if (hs == 0) {
                    uint32_t pk[8];
#pragma unroll
                    for (int e = 0; e < 16; e += 2) {
                        float dv2[2];
#pragma unroll
                        for (int u = 0; u < 2; ++u) {
                            const int j = e + u;
                            const float pr = ex2(fmaf(__uint_as_float(rm[j]), LOG2E, -lse2));
                            dv2[u] = (rowok && j < m) ? pr * (0.f - Dt) : 0.f;
                            dC[t * 16 + j] = dv2[u];
                        }
                        pk[e / 2] = f2_to_bf2(dv2[0], dv2[1]);
                    }
                    *reinterpret_cast<uint4 *>(sm + QO_DSC + 2 * TILE + sw128_offset(t, 0)) =
                        make_uint4(pk[0], pk[1], pk[2], pk[3]);
                    *reinterpret_cast<uint4 *>(sm + QO_DSC + 2 * TILE + sw128_offset(t, 16)) =
                        make_uint4(pk[4], pk[5], pk[6], pk[7]);
                }
            }
        }
        fence_proxy_async_smem();
        __syncthreads();
        // d mu[h][j][i] += sum_t dC[t][j] q[t][i]
        for (int e = tid; e < m * d; e += THREADS) {
            const int j = e / d, i = e % d;
            const uint8_t *qcol = sm + QO_Q + (i / 64) * TILE;
            float acc[4] = {0.f, 0.f, 0.f, 0.f};  // four independent partial sums over the tokens
            for (int t0 = 0; t0 < n; t0 += 4) {
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int tt = t0 + u;
                    if (tt < n)
                        acc[u] += dC[tt * 16 + j] * __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(
                                                        qcol + sw128_offset(tt, (i % 64) * 2)));
                }
            }
            atomicAdd(&a.dmu[((size_t)h * m + j) * d + i], (acc[0] + acc[1]) + (acc[2] + acc[3]));
        }
        if (!cta_wait(bar_s, 0)) break;
        tc_fence_after();
        // ---- M3: dq parts: dy S^T, tril(dA) KR, dSC [k_prev; k_cur; mu]
        if (tid == 0) {
            const uint32_t id128 = instr_desc(64, 128, FMT_BF16, 0, 0), id128b = instr_desc(64, 128, FMT_BF16, 0, 1);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                mma_bf16_ss(tmem + QT_G1, smem_desc(sb + QO_DY + (kk / 4) * TILE + (kk % 4) * 32, 16, 1024),
                            smem_desc(sb + QO_V + (kk / 4) * 2 * TILE + (kk % 4) * 32, 16, 1024), id128, kk > 0);
            if (!unsafe) {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16_ss(tmem + QT_G2, smem_desc(sb + QO_DA + kk * 32, 16, 1024),
                                smem_desc(sb + QO_KR + kk * 2048, TILE, 1024), id128b, kk > 0);
            }
            bool first = true;
            if (has_prev) {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    mma_bf16_ss(tmem + QT_DQA, smem_desc(sb + QO_DSC + kk * 32, 16, 1024),
                                smem_desc(sb + QO_KP + kk * 2048, TILE, 1024), id128b, first ? 0u : 1u);
                    first = false;
                }
            }
#pragma unroll
            for (int kk = 0; kk < 5; ++kk) {  // current chunk (kk < 4), then the 16 meta rows
                const uint32_t ao = kk < 4 ? QO_DSC + TILE + kk * 32 : QO_DSC + 2 * TILE;
                mma_bf16_ss(tmem + QT_DQA, smem_desc(sb + ao, 16, 1024),
                            smem_desc(sb + QO_KC + kk * 2048, KB_K, 1024), id128b, first ? 0u : 1u);
                first = false;
            }
            mma_commit(bar_mma);
            ++mma_issued;
        }
        if (!mma_wait()) break;
        tc_fence_after();
        // ---- E3: dq = 2^{b} dy S^T + 2^{b - r} tril(dA) KR (or the exact
        // intra-chunk sum) + dSC K; q * dq_gate
        {
            const int colh = warp >> 2;  // columns 64 colh .. 64 colh + 63
#pragma unroll 1
            for (int jj = 0; jj < 2; ++jj) {
                const int i0 = 64 * colh + 32 * jj + 16 * hs;
                uint32_t g1[16], g2[16], qa[16];
                tmem_ld16_x2<16>(tl + QT_G1 + 64 * colh + 32 * jj, g1);
                tmem_ld16_x2<16>(tl + QT_G2 + 64 * colh + 32 * jj, g2);
                tmem_ld16_x2<16>(tl + QT_DQA + 64 * colh + 32 * jj, qa);
                tmem_wait_ld();
                if (!rowok) continue;
                // gate[] = dq of the gate branch; xg[] = q * gate with the
                // intra-chunk part as QR * (tril(dA) KR), QR = bf16(q 2^{b - r})
                // rounded exactly as the key side rounds it, so that the pairs
                // that cancel in dlog gamma cancel to fp32 accuracy.
                float gate[16], xg[16];
                // The exact intra-chunk part of a wide chunk is a separate
                // copy, so that the common one holds no rare code.
                auto elems = [&](auto wide) {
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int i = i0 + e;
                        const float bt = bq[bx(t, i)];
                        const float qv = __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(
                            sm + QO_Q + (i / 64) * TILE + sw128_offset(t, (i % 64) * 2)));
                        const float inter = ex2(bt) * __uint_as_float(g1[e]);
                        gate[e] = inter;
                        xg[e] = qv * inter;
                        if constexpr (!decltype(wide)::value) {
                            const float g2v = __uint_as_float(g2[e]);
                            gate[e] += ex2(bt - rv[i]) * g2v;
                            xg[e] += __bfloat162float(__float2bfloat16_rn(qv * ex2(bt - rv[i]))) * g2v;
                        }
                    }
                    if constexpr (decltype(wide)::value) {
                        // exact: sum_{s<=t} dA[t][s] k_s[i] 2^{b_t[i] - b_s[i]} (every exponent <= 0)
                        float intra[16];
#pragma unroll
                        for (int e = 0; e < 16; ++e) intra[e] = 0.f;
                        for (int s2 = 0; s2 <= t; ++s2) {
                            const float dA = __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(
                                sm + QO_DA + sw128_offset(t, s2 * 2)));
                            if (dA == 0.f) continue;
#pragma unroll
                            for (int e = 0; e < 16; ++e) {
                                const int i = i0 + e;
                                const float kv = __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(
                                    sm + QO_KC + (i / 64) * KB_K + sw128_offset(s2, (i % 64) * 2)));
                                intra[e] += dA * kv * ex2(bq[bx(t, i)] - bq[bx(s2, i)]);
                            }
                        }
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            const int i = i0 + e;
                            const float qv = __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(
                                sm + QO_Q + (i / 64) * TILE + sw128_offset(t, (i % 64) * 2)));
                            gate[e] += intra[e];
                            xg[e] += qv * intra[e];
                        }
                    }
                };
                if (!unsafe)
                    elems(std::false_type{});
                else
                    elems(std::true_type{});
                const size_t row = (size_t)unit * L + c0 + t;
                uint32_t pk[8];
#pragma unroll
                for (int e = 0; e < 16; e += 2)
                    pk[e / 2] = f2_to_bf2(gate[e] + __uint_as_float(qa[e]), gate[e + 1] + __uint_as_float(qa[e + 1]));
                if (i0 < d) {
                    uint4 *dqp = reinterpret_cast<uint4 *>(a.dq + row * d + i0);
                    dqp[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                    dqp[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
                }
                float4 *xqp = reinterpret_cast<float4 *>(a.xq + row * D + i0);
#pragma unroll
                for (int u = 0; u < 4; ++u) xqp[u] = make_float4(xg[4 * u], xg[4 * u + 1], xg[4 * u + 2], xg[4 * u + 3]);
            }
        }
    } while (false);
    // Drain (bounded) before shared and tensor memory are released.
    if (tid == 0) {
        for (uint32_t i = mma_use; i < mma_issued; ++i)
            if (!mbar_wait(bar_mma, i & 1u, WAIT)) break;
        if (in_issued) mbar_wait(bar_in, 0, WAIT);
        if (s_issued) mbar_wait(bar_s, 0, WAIT);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

// ============================================================ key side
struct KeyArgs {
    const __nv_bfloat16 *Sb;      // [units][nchunks][D][D]  state before chunk c
    const float *xq;              // [units][L][D]  q * dq_gate
    const float *lse2, *drow;     // [units][L]
    __nv_bfloat16 *dk, *dv, *dg;  // [units][L][D]  (dk, dv per query head; summed over a group afterwards)
    float alpha;
    int L, w, nchunks;
    const float *alpha_h;         // per-head anchor weights (null: alpha)
    int H, group;                 // query heads per key/value head
};

// Shared memory of bwd_key_kernel.  Phase A (anchor products) uses the
// next chunk's q/dy and four probability tiles; phase B (gate products)
// reuses those slots for b, QR, KR/KL.
constexpr uint32_t KO_Q = 0, KO_K = KO_Q + 2 * TILE, KO_V = KO_K + 2 * TILE, KO_DY = KO_V + 2 * TILE;
constexpr uint32_t KO_G = KO_DY + 2 * TILE;
constexpr uint32_t KO_QN = KO_G + 2 * TILE;     // q of the next chunk; phase B: QR = q 2^{b - r}
constexpr uint32_t KO_DYN = KO_QN + 2 * TILE;   // dy of the next chunk; phase B: KR = k 2^{r - b}, then KL
constexpr uint32_t KO_H = KO_DYN + 2 * TILE;    // state gradient after the chunk [128][128]
constexpr uint32_t KO_PC = KO_H + 4 * TILE;     // alpha P (this chunk's rows) [t][s]; phase B: b fp32 (4 tiles)
constexpr uint32_t KO_DSCC = KO_PC + TILE;      // score gradients, this chunk's rows
constexpr uint32_t KO_PN = KO_DSCC + TILE;      // alpha P, next chunk's rows
constexpr uint32_t KO_DSCN = KO_PN + TILE;      // score gradients, next chunk's rows
constexpr uint32_t KO_DAT = KO_DSCN + TILE;     // tril(dy v^T) [t][s]
constexpr uint32_t KO_AT = KO_DAT + TILE;       // tril(A) [t][s]
constexpr uint32_t KO_B = KO_PC;
constexpr uint32_t KO_VEC = KO_AT + TILE;       // r[128], b_last[128], tot[4][128], E parts [2][128]
constexpr uint32_t KO_BAR = KO_VEC + (128 + 128 + 512 + 256) * 4;
constexpr uint32_t KO_TSLOT = KO_BAR + 3 * 8;
constexpr uint32_t KO_SMEM = KO_TSLOT + 8 + 1024;
static_assert(KO_SMEM <= 232448, "shared memory budget");
// Tensor-memory columns: phase A scores / dy v^T, anchor dk / dv; phase B
// A, then the two gate parts of dk (dv accumulates on).
constexpr uint32_t KT_SCC = 0, KT_DA = 64, KT_SCN = 128, KT_DPN = 192, KT_DKA = 256, KT_DV = 384;
constexpr uint32_t KT_A = 0, KT_G1 = 0, KT_G2 = 128;

template <int DH>
__global__ void __launch_bounds__(THREADS, 1)
    bwd_key_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                   const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tg,
                   const __grid_constant__ CUtensorMap tdy, const __grid_constant__ CUtensorMap tH,
                   const KeyArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = smem_align1024(smem_raw);
    const uint32_t sb = smem_u32(sm);
    float *rv = reinterpret_cast<float *>(sm + KO_VEC), *blv = rv + 128, *tot = blv + 128, *Ep = tot + 512;
    float *bk = reinterpret_cast<float *>(sm + KO_B);  // phase B: b [64][128]
    float *yo = reinterpret_cast<float *>(sm + KO_QN);  // after the gate products: k * dk_inter [64][128]
    // Element (t, i) of bk / yo sits at column i ^ (t mod 32) of row t, so
    // that a warp reading one column of 16 rows (two column halves) hits 32
    // distinct banks; a row read along i stays a permutation of one row.
    auto bx = [](int t, int i) { return t * D + (i ^ (t & 31)); };
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + KO_BAR);
    uint64_t *bar_in = bars, *bar_mma = bars + 1;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + KO_TSLOT);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nch = a.nchunks;
    const int unit = blockIdx.x / nch, c = blockIdx.x % nch;
    const int L = a.L, w = a.w;
    const int c0 = c * C, n = min(C, L - c0);
    const bool has_next = c + 1 < nch;
    const int nn = has_next ? min(C, L - c0 - C) : 0;  // rows of the next chunk
    const float alpha = head_alpha(a.alpha_h, a.alpha, unit % a.H);
    const int kvu = kv_unit(unit, a.H, a.group);

    constexpr int d = DH, nbox = DH / 64;
    if constexpr (DH < D) {
        // block 1 of q, k, v, dy, g and of the next chunk's q, dy
        const uint32_t blk[7] = {KO_Q + TILE, KO_K + TILE, KO_V + TILE, KO_DY + TILE, KO_G + TILE, KO_QN + TILE,
                                 KO_DYN + TILE};
        clear_blocks(sm, blk, TILE);
        fence_proxy_async_smem();
    }
    if (warp == 0) {
        tmem_alloc(tslot, 512);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(bar_in, 1);
        mbar_init(bar_mma, 1);
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    uint32_t mma_use = 0, mma_issued = 0, in_issued = 0;
    if (tid == 0) {
        mbar_arrive_expect_tx(bar_in, ((has_next ? 7 : 5) * nbox + 4) * TILE);
        for (int hb = 0; hb < 2; ++hb) {
            for (int ib = 0; ib < 2; ++ib)
                tma_load_3d(sm + KO_H + hb * 2 * TILE + ib * TILE, &tH, bar_in, 64 * hb, 64 * ib, unit * nch + c);
            if (hb >= nbox) continue;
            tma_load_3d(sm + KO_Q + hb * TILE, &tq, bar_in, 64 * hb, c0, unit);
            tma_load_3d(sm + KO_K + hb * TILE, &tk, bar_in, 64 * hb, c0, kvu);
            tma_load_3d(sm + KO_V + hb * TILE, &tv, bar_in, 64 * hb, c0, kvu);
            tma_load_3d(sm + KO_DY + hb * TILE, &tdy, bar_in, 64 * hb, c0, unit);
            tma_load_3d(sm + KO_G + hb * TILE, &tg, bar_in, 64 * hb, c0, unit);
            if (has_next) {
                tma_load_3d(sm + KO_QN + hb * TILE, &tq, bar_in, 64 * hb, c0 + C, unit);
                tma_load_3d(sm + KO_DYN + hb * TILE, &tdy, bar_in, 64 * hb, c0 + C, unit);
            }
        }
        in_issued = 1;
    }
    auto mma_wait = [&]() -> bool {
        const bool r = cta_wait(bar_mma, mma_use);
        if (r) ++mma_use;
        return r;
    };
    auto commit = [&]() {
        mma_commit(bar_mma);
        ++mma_issued;
    };
    const int quarter = warp & 3, hs = lane >> 4;
    const int t = 16 * quarter + (lane & 15);  // this thread's accumulator row
    const uint32_t tl = tmem + tlane(quarter);
    // row statistics of this thread's query row (warps 0-3: this chunk,
    // warps 4-7: the next chunk), fetched while the tiles load
    const bool nxt = warp >= 4;
    const int tq_row = nxt ? c0 + C + t : c0 + t;
    const bool qrow_ok = nxt ? t < nn : t < n;
    const float l2 = qrow_ok ? a.lse2[(size_t)unit * L + tq_row] : 0.f;
    const float Dt = qrow_ok ? a.drow[(size_t)unit * L + tq_row] : 0.f;
    // The state before this chunk, row i = tid % 128, columns 64 (tid / 128)
    // .. + 63, fetched while the tiles load (for the later chunks' share of
    // dlog gamma below).
    uint4 sv[8];
    {
        const uint4 *Sp = reinterpret_cast<const uint4 *>(a.Sb + ((size_t)unit * nch + c) * D * D +
                                                          (size_t)(tid & 127) * D + 64 * (tid >> 7));
#pragma unroll
        for (int u = 0; u < 8; ++u) sv[u] = ldg_early(Sp + u);
    }
    int unsafe = 0;
    do {
        if (!cta_wait(bar_in, 0)) break;
        // ---- M1a: this chunk's rows and the next chunk's rows against this chunk's keys
        if (tid == 0) {
            const uint32_t id64 = instr_desc(64, 64, FMT_BF16, 0, 0);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint32_t ko = (kk / 4) * TILE + (kk % 4) * 32;
                const uint64_t kd = smem_desc(sb + KO_K + ko, 16, 1024), vd = smem_desc(sb + KO_V + ko, 16, 1024);
                mma_bf16_ss(tmem + KT_SCC, smem_desc(sb + KO_Q + ko, 16, 1024), kd, id64, kk > 0);
                mma_bf16_ss(tmem + KT_DA, smem_desc(sb + KO_DY + ko, 16, 1024), vd, id64, kk > 0);
                if (has_next) {
                    mma_bf16_ss(tmem + KT_SCN, smem_desc(sb + KO_QN + ko, 16, 1024), kd, id64, kk > 0);
                    mma_bf16_ss(tmem + KT_DPN, smem_desc(sb + KO_DYN + ko, 16, 1024), vd, id64, kk > 0);
                }
            }
            commit();
        }
        // the later chunks' share of dlog gamma needs sum_j Sb[c][i][j] H[i][j]
        // (scaled by 2^{b_last} later): row i, columns 64 half .. + 63
        {
            const int i = tid & 127, half = tid >> 7;
            float acc = 0.f;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const uint4 hv = *reinterpret_cast<const uint4 *>(sm + KO_H + half * 2 * TILE + sw128_offset(i, 16 * u));
                const uint32_t sw[4] = {sv[u].x, sv[u].y, sv[u].z, sv[u].w}, hw[4] = {hv.x, hv.y, hv.z, hv.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 s2 = bf2_to_f2(sw[e]), h2 = bf2_to_f2(hw[e]);
                    acc = fmaf(s2.x, h2.x, acc);
                    acc = fmaf(s2.y, h2.y, acc);
                }
            }
            Ep[half * 128 + i] = acc;
        }
        if (!mma_wait()) break;
        tc_fence_after();
        // ---- E1a: probabilities and score gradients (warps 0-3: this chunk's
        // rows; warps 4-7: the next chunk's rows), tril(dy v^T)
        {
            const int tg = tq_row;  // query position
            const bool rowok = qrow_ok;
            // key s of this chunk is in row tg's window iff tg - w + 1 <= c0 + s <= tg
            const int slo = tg - w + 1 - c0, shi = tg - c0;
            uint32_t r[2][16], d[2][16];
            tmem_ld16_x2<16>(tl + (nxt ? KT_SCN : KT_SCC), r[0]);
            tmem_ld16_x2<16>(tl + (nxt ? KT_SCN : KT_SCC) + 32, r[1]);
            tmem_ld16_x2<16>(tl + (nxt ? KT_DPN : KT_DA), d[0]);
            tmem_ld16_x2<16>(tl + (nxt ? KT_DPN : KT_DA) + 32, d[1]);
            tmem_wait_ld();
            const uint32_t op = nxt ? KO_PN : KO_PC, od = nxt ? KO_DSCN : KO_DSCC;
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
                const int s0 = 32 * jj + 16 * hs;
                uint32_t pp[8], pd[8], pa[8];
#pragma unroll
                for (int e = 0; e < 16; e += 2) {
                    float vp[2], vd[2], va[2];
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int s2 = s0 + e + u;
                        const bool valid = rowok && s2 >= slo && s2 <= shi && s2 < n;
                        const float pr = ex2(fmaf(__uint_as_float(r[jj][e + u]), LOG2E, -l2));
                        const float dp = __uint_as_float(d[jj][e + u]);
                        vp[u] = valid ? alpha * pr : 0.f;
                        vd[u] = valid ? pr * (alpha * dp - Dt) : 0.f;
                        va[u] = (!nxt && rowok && s2 <= t) ? dp : 0.f;
                    }
                    pp[e / 2] = f2_to_bf2(vp[0], vp[1]);
                    pd[e / 2] = f2_to_bf2(vd[0], vd[1]);
                    pa[e / 2] = f2_to_bf2(va[0], va[1]);
                }
                const uint32_t o0 = sw128_offset(t, s0 * 2), o1 = sw128_offset(t, s0 * 2 + 16);
                *reinterpret_cast<uint4 *>(sm + op + o0) = make_uint4(pp[0], pp[1], pp[2], pp[3]);
                *reinterpret_cast<uint4 *>(sm + op + o1) = make_uint4(pp[4], pp[5], pp[6], pp[7]);
                *reinterpret_cast<uint4 *>(sm + od + o0) = make_uint4(pd[0], pd[1], pd[2], pd[3]);
                *reinterpret_cast<uint4 *>(sm + od + o1) = make_uint4(pd[4], pd[5], pd[6], pd[7]);
                if (!nxt) {
                    *reinterpret_cast<uint4 *>(sm + KO_DAT + o0) = make_uint4(pa[0], pa[1], pa[2], pa[3]);
                    *reinterpret_cast<uint4 *>(sm + KO_DAT + o1) = make_uint4(pa[4], pa[5], pa[6], pa[7]);
                }
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        // ---- M2a: anchor dk = dSC^T q, dv = alpha P^T dy (both row blocks)
        if (tid == 0) {
            const uint32_t idmm = instr_desc(64, 128, FMT_BF16, 1, 1);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                mma_bf16_ss(tmem + KT_DKA, smem_desc(sb + KO_DSCC + kk * 2048, TILE, 1024),
                            smem_desc(sb + KO_Q + kk * 2048, TILE, 1024), idmm, kk > 0);
                mma_bf16_ss(tmem + KT_DV, smem_desc(sb + KO_PC + kk * 2048, TILE, 1024),
                            smem_desc(sb + KO_DY + kk * 2048, TILE, 1024), idmm, kk > 0);
            }
            if (has_next) {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    mma_bf16_ss(tmem + KT_DKA, smem_desc(sb + KO_DSCN + kk * 2048, TILE, 1024),
                                smem_desc(sb + KO_QN + kk * 2048, TILE, 1024), idmm, 1u);
                    mma_bf16_ss(tmem + KT_DV, smem_desc(sb + KO_PN + kk * 2048, TILE, 1024),
                                smem_desc(sb + KO_DYN + kk * 2048, TILE, 1024), idmm, 1u);
                }
            }
            commit();
        }
        if (!mma_wait()) break;
        // ---- prep (phase B): b, r = b at token 31, QR, KR; the probability
        // tiles and the next chunk's tiles are free now
        {
            const int p = tid & 63, hq = tid >> 6;
            Prefix pf;
            local_prefix(sm + KO_G, p, hq, n, pf, tot);
            __syncthreads();
            const float2 bl = finish_prefix(p, hq, pf, tot);
            if (hq == 1) {
                rv[2 * p] = pf.b[15].x;
                rv[2 * p + 1] = pf.b[15].y;
            }
            if (hq == 0) {
                blv[2 * p] = bl.x;
                blv[2 * p + 1] = bl.y;
            }
            __syncthreads();
            const float2 r2 = make_float2(rv[2 * p], rv[2 * p + 1]);
            const uint32_t kblk = (p / 32) * TILE, kbyte = (p % 32) * 4;
            bool wide = false;
#pragma unroll
            for (int tt = 0; tt < 16; ++tt) {
                const int t2 = 16 * hq + tt;
                const float2 bt = pf.b[tt];
                wide |= fabsf(bt.x - r2.x) > SPAN2_MAX || fabsf(bt.y - r2.y) > SPAN2_MAX;
                bk[bx(t2, 2 * p)] = bt.x;
                bk[bx(t2, 2 * p + 1)] = bt.y;
                const uint32_t o = kblk + sw128_offset(t2, kbyte);
                const float2 qv = bf2_to_f2(*reinterpret_cast<const uint32_t *>(sm + KO_Q + o));
                const float2 kv = bf2_to_f2(*reinterpret_cast<const uint32_t *>(sm + KO_K + o));
                *reinterpret_cast<uint32_t *>(sm + KO_QN + o) =
                    f2_to_bf2(qv.x * ex2(bt.x - r2.x), qv.y * ex2(bt.y - r2.y));
                *reinterpret_cast<uint32_t *>(sm + KO_DYN + o) =
                    f2_to_bf2(kv.x * ex2(r2.x - bt.x), kv.y * ex2(r2.y - bt.y));
            }
            unsafe = __syncthreads_or(wide);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        // ---- M1b: A = QR KR^T
        if (tid == 0) {
            if (!unsafe) {
                const uint32_t id64 = instr_desc(64, 64, FMT_BF16, 0, 0);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t ko = (kk / 4) * TILE + (kk % 4) * 32;
                    mma_bf16_ss(tmem + KT_A, smem_desc(sb + KO_QN + ko, 16, 1024),
                                smem_desc(sb + KO_DYN + ko, 16, 1024), id64, kk > 0);
                }
            }
            commit();
        }
        if (!mma_wait()) break;
        tc_fence_after();
        // ---- E1b: tril(A) (exact on the CUDA cores for a wide chunk); KL = k 2^{b_last - b}
        {
            if (warp < 4) {
                uint32_t r[2][16];
                tmem_ld16_x2<16>(tl + KT_A, r[0]);
                tmem_ld16_x2<16>(tl + KT_A + 32, r[1]);
                tmem_wait_ld();
                if (!unsafe) {
#pragma unroll
                    for (int jj = 0; jj < 2; ++jj) {
                        const int s0 = 32 * jj + 16 * hs;
                        uint32_t pk[8];
#pragma unroll
                        for (int e = 0; e < 16; e += 2)
                            pk[e / 2] = f2_to_bf2(t < n && s0 + e <= t ? __uint_as_float(r[jj][e]) : 0.f,
                                                  t < n && s0 + e + 1 <= t ? __uint_as_float(r[jj][e + 1]) : 0.f);
                        *reinterpret_cast<uint4 *>(sm + KO_AT + sw128_offset(t, s0 * 2)) =
                            make_uint4(pk[0], pk[1], pk[2], pk[3]);
                        *reinterpret_cast<uint4 *>(sm + KO_AT + sw128_offset(t, s0 * 2 + 16)) =
                            make_uint4(pk[4], pk[5], pk[6], pk[7]);
                    }
                } else {
                    // exact, one score at a time (a rare path: small code)
#pragma unroll 1
                    for (int sx = 0; sx < 32; ++sx) {
                        const int s2 = 32 * (sx / 16) + 16 * hs + sx % 16;
                        float av = 0.f;
                        if (t < n && s2 <= t) {
#pragma unroll 1
                            for (int i = 0; i < D; ++i) {
                                const uint32_t ob = (i / 64) * TILE;
                                const float qv = __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(
                                    sm + KO_Q + ob + sw128_offset(t, (i % 64) * 2)));
                                const float kv = __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(
                                    sm + KO_K + ob + sw128_offset(s2, (i % 64) * 2)));
                                av += qv * kv * ex2(bk[bx(t, i)] - bk[bx(s2, i)]);
                            }
                        }
                        *reinterpret_cast<__nv_bfloat16 *>(sm + KO_AT + sw128_offset(t, s2 * 2)) = __float2bfloat16_rn(av);
                    }
                }
            }
            {
                // KL into the KR slot (KR was read by M1b, which is done)
                for (int e = tid; e < C * 64; e += THREADS) {
                    const int s2 = e / 64, ip = e % 64, i = 2 * ip;
                    const uint32_t o = (i / 64) * TILE + sw128_offset(s2, (i % 64) * 2);
                    const float2 kv = bf2_to_f2(*reinterpret_cast<const uint32_t *>(sm + KO_K + o));
                    const float bl0 = bk[bx(C - 1, i)], bl1 = bk[bx(C - 1, i + 1)];
                    *reinterpret_cast<uint32_t *>(sm + KO_DYN + o) =
                        f2_to_bf2(kv.x * ex2(bl0 - bk[bx(s2, i)]), kv.y * ex2(bl1 - bk[bx(s2, i + 1)]));
                }
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        // ---- M2b: dk gate parts V H^T, tril(dA)^T QR; dv += KL H + tril(A)^T dy
        if (tid == 0) {
            const uint32_t idkk = instr_desc(64, 128, FMT_BF16, 0, 0), idmm = instr_desc(64, 128, FMT_BF16, 1, 1);
            const uint32_t idkm = instr_desc(64, 128, FMT_BF16, 0, 1);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                mma_bf16_ss(tmem + KT_G1, smem_desc(sb + KO_V + (kk / 4) * TILE + (kk % 4) * 32, 16, 1024),
                            smem_desc(sb + KO_H + (kk / 4) * 2 * TILE + (kk % 4) * 32, 16, 1024), idkk, kk > 0);
                mma_bf16_ss(tmem + KT_DV, smem_desc(sb + KO_DYN + (kk / 4) * TILE + (kk % 4) * 32, 16, 1024),
                            smem_desc(sb + KO_H + kk * 2048, 2 * TILE, 1024), idkm, 1u);
            }
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                if (!unsafe)
                    mma_bf16_ss(tmem + KT_G2, smem_desc(sb + KO_DAT + kk * 2048, TILE, 1024),
                                smem_desc(sb + KO_QN + kk * 2048, TILE, 1024), idmm, kk > 0);
                mma_bf16_ss(tmem + KT_DV, smem_desc(sb + KO_AT + kk * 2048, TILE, 1024),
                            smem_desc(sb + KO_DY + kk * 2048, TILE, 1024), idmm, 1u);
            }
            commit();
        }
        // q * dq_gate of this thread's row and columns, fetched while the
        // gate products run
        uint4 xq4[2][4];
        if (t < n) {
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
                const float4 *xp = reinterpret_cast<const float4 *>(
                    a.xq + ((size_t)unit * L + c0 + t) * D + 64 * (warp >> 2) + 32 * jj + 16 * hs);
#pragma unroll
                for (int u = 0; u < 4; ++u) xq4[jj][u] = ldg_early(xp + u);
            }
        }
        if (!mma_wait()) break;
        tc_fence_after();
        // ---- E2: dk, dv; the dlog gamma terms.  With dk_gate = dk_inter +
        // dk_intra, the later chunks' share (sum_j S_after H) minus the
        // k * dk_inter of this chunk's tokens >= t is 2^{b_last} sum_j Sb H
        // plus the k * dk_inter of its tokens < t, so
        //   dlog gamma_t = sum_{r>=t} (q dq_gate - k dk_intra)_r + E + sum_{s<t} (k dk_inter)_s,
        //   E[i] = 2^{b_last[i]} sum_j Sb[c][i][j] H[i][j],
        // and k dk_intra uses KR = bf16(k 2^{r - b}) as the query side uses
        // QR, so that the pairs inside the suffix cancel to fp32 accuracy.
        {
            const int colh = warp >> 2;
            const bool rowok = t < n;
            const size_t row = (size_t)unit * L + c0 + t;
            float term[2][16];
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
                const int i0 = 64 * colh + 32 * jj + 16 * hs;
                const uint32_t cofs = 64 * colh + 32 * jj;
                uint32_t g1[16], g2[16], ka[16], vv[16];
                float xqv[16];
                if (rowok) {
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const uint4 x4 = xq4[jj][u];
                        xqv[4 * u] = __uint_as_float(x4.x);
                        xqv[4 * u + 1] = __uint_as_float(x4.y);
                        xqv[4 * u + 2] = __uint_as_float(x4.z);
                        xqv[4 * u + 3] = __uint_as_float(x4.w);
                    }
                }
                tmem_ld16_x2<16>(tl + KT_G1 + cofs, g1);
                tmem_ld16_x2<16>(tl + KT_G2 + cofs, g2);
                tmem_ld16_x2<16>(tl + KT_DKA + cofs, ka);
                tmem_ld16_x2<16>(tl + KT_DV + cofs, vv);
                tmem_wait_ld();
                uint32_t dkp[8], dvp[8];
                float dkv[16];
                // The exact intra-chunk part of a wide chunk is a separate
                // copy of the loop, so that the common one holds no rare code.
                auto elems = [&](auto wide) {
                    // shared-memory reads first, writes last: nothing in
                    // between waits on an aliasing store
                    float bsv[16], kvv[16], yov[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int i = i0 + e;
                        bsv[e] = rowok ? bk[bx(t, i)] : 0.f;
                        kvv[e] = rowok ? __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(
                                             sm + KO_K + (i / 64) * TILE + sw128_offset(t, (i % 64) * 2)))
                                       : 0.f;
                    }
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int i = i0 + e;
                        const float bs = bsv[e], kv = kvv[e];
                        const float inter = ex2(blv[i] - bs) * __uint_as_float(g1[e]);
                        float intra = 0.f, kintra = 0.f;
                        if constexpr (!decltype(wide)::value) {
                            const float g2v = __uint_as_float(g2[e]);
                            const float sc = ex2(rv[i] - bs);
                            intra = sc * g2v;
                            kintra = __bfloat162float(__float2bfloat16_rn(kv * sc)) * g2v;
                        } else {
                            if (rowok) {
#pragma unroll 1
                                for (int t2 = t; t2 < n; ++t2) {
                                    const float dA = __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(
                                        sm + KO_DAT + sw128_offset(t2, t * 2)));
                                    const float qv = __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(
                                        sm + KO_Q + (i / 64) * TILE + sw128_offset(t2, (i % 64) * 2)));
                                    intra += dA * qv * ex2(bk[bx(t2, i)] - bs);
                                }
                            }
                            kintra = kv * intra;
                        }
                        dkv[e] = rowok ? inter + intra + __uint_as_float(ka[e]) : 0.f;
                        term[jj][e] = rowok ? xqv[e] - kintra : 0.f;
                        yov[e] = rowok ? kv * inter : 0.f;
                    }
#pragma unroll
                    for (int e = 0; e < 16; ++e) yo[bx(t, i0 + e)] = yov[e];  // the QR / KL slot: M2b is done
                };
                if (!unsafe)
                    elems(std::false_type{});
                else
                    elems(std::true_type{});
#pragma unroll
                for (int e = 0; e < 16; e += 2) {
                    dkp[e / 2] = f2_to_bf2(dkv[e], dkv[e + 1]);
                    dvp[e / 2] = f2_to_bf2(__uint_as_float(vv[e]), __uint_as_float(vv[e + 1]));
                }
                if (rowok && i0 < d) {
                    uint4 *dkq = reinterpret_cast<uint4 *>(a.dk + row * d + i0);
                    uint4 *dvq = reinterpret_cast<uint4 *>(a.dv + row * d + i0);
                    dkq[0] = make_uint4(dkp[0], dkp[1], dkp[2], dkp[3]);
                    dkq[1] = make_uint4(dkp[4], dkp[5], dkp[6], dkp[7]);
                    dvq[0] = make_uint4(dvp[0], dvp[1], dvp[2], dvp[3]);
                    dvq[1] = make_uint4(dvp[4], dvp[5], dvp[6], dvp[7]);
                }
            }
            __syncthreads();  // every read of b is done
#pragma unroll
            for (int jj = 0; jj < 2; ++jj)
#pragma unroll
                for (int e = 0; e < 16; ++e) bk[bx(t, 64 * colh + 32 * jj + 16 * hs + e)] = term[jj][e];
        }
        // ---- dg = dlog gamma * sigmoid(-g).  sigmoid(-g) = 2^{log2 sigmoid(-g)}
        // for every element first (into the state-gradient slot: its readers
        // are done), then two threads per column scan half a chunk each.
        __syncthreads();  // the terms and k dk_inter of every row are written
        float *sg = reinterpret_cast<float *>(sm + KO_H);
        for (int e = tid; e < C * 64; e += THREADS) {
            const int t2 = e / 64, ip = e % 64, i = 2 * ip;
            const float2 gv = bf2_to_f2(*reinterpret_cast<const uint32_t *>(
                sm + KO_G + (i / 64) * TILE + sw128_offset(t2, (i % 64) * 2)));
            sg[t2 * D + i] = ex2(log2_sigmoid(-gv.x));
            sg[t2 * D + i + 1] = ex2(log2_sigmoid(-gv.y));
        }
        float *part = Ep;  // [2][128]: the upper half's sum of terms, the lower half's sum of k dk_inter
        const int i = tid & 127, half = tid >> 7;
        const int h0 = half * (C / 2), h1 = min(n, h0 + C / 2);
        {
            float sr = 0.f, sf = 0.f;
#pragma unroll 8
            for (int t2 = h0; t2 < h1; ++t2) {
                sr += bk[bx(t2, i)];
                sf += yo[bx(t2, i)];
            }
            __syncthreads();  // Ep (the E parts) is read below, before it is reused
            const float E = (Ep[i] + Ep[128 + i]) * ex2(blv[i]);
            __syncthreads();
            if (half == 1) part[i] = sr;        // terms of rows 32 .. 63, for the reverse prefix of rows < 32
            if (half == 0) part[128 + i] = sf;  // k dk_inter of rows 0 .. 31, for the forward prefix of rows >= 32
            __syncthreads();
            float run = (half == 0 ? part[i] : 0.f) + E;  // reverse: later rows first
            float f = half == 1 ? part[128 + i] : 0.f;   // forward exclusive prefix
#pragma unroll 8
            for (int t2 = h0; t2 < h1; ++t2) {  // forward prefix of k dk_inter, in place
                const float x = yo[bx(t2, i)];
                yo[bx(t2, i)] = f;
                f += x;
            }
#pragma unroll 8
            for (int t2 = h1 - 1; t2 >= h0; --t2) {
                run += bk[bx(t2, i)];
                if (i < d)
                    a.dg[((size_t)unit * L + c0 + t2) * d + i] =
                        __float2bfloat16_rn((run + yo[bx(t2, i)]) * sg[t2 * D + i]);
            }
        }
    } while (false);
    if (tid == 0) {
        for (uint32_t i = mma_use; i < mma_issued; ++i)
            if (!mbar_wait(bar_mma, i & 1u, WAIT)) break;
        if (in_issued) mbar_wait(bar_in, 0, WAIT);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

}  // namespace bwdtc
}  // namespace lizard
