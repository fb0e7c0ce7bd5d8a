// prefill_tc.cuh -- chunked Lizard prefill on tcgen05 tensor cores (bf16, d = 128).
//
// Operator: gated linear attention (Lizard, gist.science/de section 2 item 1)
// + anchor window with meta-memory sinks (item 2) + alpha combine (item 3).
// The chunked, log-space form follows the page's "Hardware-bewusster
// Algorithmus" section: cumulative gate terms are kept as log-space prefix
// sums and folded into the query/key operands so that the intra-chunk work
// becomes plain GEMMs on the tensor cores.
//
// One CTA walks the chunks (C = 64 tokens) of one (batch, head) sequence.
// Per chunk, with b_t = sum_{r=c0..t} log sigmoid(g_r) (per key dim, fp32,
// base-2 internally) and the chunk reference r = (b_c0 + b_last) / 2:
//
//   scores  [t, s'] = q_t . k_s'  (band of the previous ceil((w-1)/64) chunks
//                     and this one) and q_t . mu_j        tcgen05, M=64
//   A       [t, s]  = (q * e^{b-r})_t . (k * e^{r-b})_s   tcgen05, M=64
//   W       [t, s'] = alpha * softmax-with-sinks(scores) + A (s' in chunk, s <= t)
//   y^T     [j, t]  = S^T (TMEM, tf32) . (q * e^{b})^T + V_band^T . W^T
//   S^T    <- S^T * diag(e^{b_last}) + V^T . (k * e^{b_last - b})
//
// Exponent ranges.  e^{b} and e^{b_last-b} have exponents <= 0.  The two
// factors of A have exponents within +-(b_c0 - b_last)/2, which is kept
// within +-SPAN_HALF_MAX nats so that neither factor leaves the normal bf16
// range for any |q|, |k| above 1e-7.  A chunk whose decay span exceeds that
// for any key dimension computes A exactly on the CUDA cores instead
// (sum_i q k e^{b_t-b_s}, exponent <= 0) and stores it into tensor memory;
// the rest of the chunk is unchanged.  So every gate value is handled.
//
// Layouts.  Shared-memory operand tiles are 128B-swizzled (K-major: rows of
// 128 B along K; the v tile as loaded is the MN-major operand of the two
// V^T products).  Tensor memory (512 columns):
//   [0,128)   S^T  fp32, lane = value dim j, column = key dim i
//   [128,336) scores, M=64 layout (row t in lane 32(t/16) + t%16): 16 meta
//             columns, then 64 per band chunk
//   [336,400) A (M=64 layout), later y^T part 2 (M=128, lane = j)
//   [400,464) y^T part 1 (tf32 product with the state)
#pragma once

#include "common.cuh"
#include "sm100.cuh"

namespace lizard {
namespace tc {

using namespace sm100;

constexpr int C = 64;
constexpr int D = 128;
constexpr int THREADS = 256;
constexpr int NR = 4;                   // k/v ring slots (band of 2 previous chunks + current + prefetch)
constexpr int MAX_PREV = 2;             // previous chunks in the band: w <= 129
constexpr int META_ROWS = 16;
constexpr float LOG2E = 1.4426950408889634f;
// Largest exponent magnitude (nats) of the two intra-chunk factors.
constexpr float SPAN_HALF_MAX = 72.f;
constexpr float SPAN_MAX2 = 2.f * SPAN_HALF_MAX * LOG2E;   // chunk decay span limit, base 2

// Shared-memory map (offsets from a 1024-aligned base).
constexpr uint32_t TILE = C * 128;                 // one 64-row x 128-byte swizzled block: 8 KB
constexpr uint32_t OFF_Q = 0;                      // q tile: 2 blocks (16 KB)
constexpr uint32_t OFF_KV = OFF_Q + 2 * TILE;      // NR slots x (k 16 KB + v 16 KB)
constexpr uint32_t KV_SLOT = 4 * TILE;
constexpr uint32_t V_OFF = 2 * TILE;               // v tile within a slot
constexpr uint32_t OFF_QZ = OFF_KV + NR * KV_SLOT; // 32 KB: QR (bf16) | q*e^{b} (fp32) | exact-A scratch
constexpr uint32_t OFF_KW = OFF_QZ + 4 * TILE;     // 24 KB: KR (bf16) | W (bf16, up to 192 columns)
constexpr uint32_t OFF_KL = OFF_KW + 3 * TILE;     // 16 KB: k * e^{b_last - b} (bf16)
constexpr uint32_t OFF_MU = OFF_KL + 2 * TILE;     // 4 KB: meta keys, 16 rows x 128
constexpr uint32_t MU_BLOCK = META_ROWS * 128;
constexpr uint32_t OFF_VEC = OFF_MU + 2 * MU_BLOCK;
constexpr uint32_t VEC_FLOATS = 4 * 128 + 4 * 64;  // xch, first, last, dec, red[2][2][64]
constexpr uint32_t OFF_BAR = OFF_VEC + VEC_FLOATS * 4;
constexpr uint32_t NBARS = 1 + NR + 3;
constexpr uint32_t SMEM_USED = OFF_BAR + NBARS * 8 + 16;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;  // alignment slack
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

// Tensor-memory columns.
constexpr uint32_t T_ST = 0, T_SC = 128, T_A = 336, T_Y2 = 336, T_Y1 = 400, T_COLS = 512;

constexpr uint32_t WAIT_LIMIT = 1u << 21;

struct TcArgs {
    const __nv_bfloat16 *g, *mu, *k, *v;
    __nv_bfloat16 *y;
    float *S_out;
    __nv_bfloat16 *ring_k, *ring_v;
    int64_t *pos;
    float alpha;
    int H, L, w, m, nprev;
};

__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float lg2(float x)
{
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// log2(sigmoid(g)) = min(g, 0) log2(e) - log2(1 + 2^{-|g| log2(e)})
__device__ __forceinline__ float log2_sigmoid(float g)
{
    return fminf(g, 0.f) * LOG2E - lg2(1.f + ex2(-fabsf(g) * LOG2E));
}

__device__ __forceinline__ uint32_t tmem_lane(uint32_t quarter) { return (32u * quarter) << 16; }

__device__ __forceinline__ __nv_bfloat16 ld_bf16(const uint8_t *p) { return *reinterpret_cast<const __nv_bfloat16 *>(p); }
__device__ __forceinline__ void st_bf16(uint8_t *p, float x) { *reinterpret_cast<__nv_bfloat16 *>(p) = __float2bfloat16_rn(x); }

__global__ void __launch_bounds__(THREADS, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                      const __grid_constant__ CUtensorMap tv, const TcArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(sm);
    float *xch = reinterpret_cast<float *>(sm + OFF_VEC);
    float *first2 = xch + 128, *last2 = first2 + 128, *dec = last2 + 128;
    float *red = dec + 128;  // [pass 2][half 2][row 64]
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + OFF_BAR);
    uint64_t *bar_q = bars, *bar_kv = bars + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + NBARS);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3, half = warp >> 2;
    const int unit = blockIdx.x, h = unit % a.H;
    const int L = a.L, NP = a.nprev, w = a.w, m = a.m;
    const int nchunks = (L + C - 1) / C;
    const int gi = tid & 127, gth = tid >> 7;  // prep: key dim and token half

    if (warp == 0) {
        tmem_alloc(tmem_slot, T_COLS);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (uint32_t i = 0; i < NBARS; ++i) mbar_init(&bars[i], 1);
        fence_mbar_init();
        prefetch_tmap(&tq);
        prefetch_tmap(&tk);
        prefetch_tmap(&tv);
    }
    // Meta keys of this head, zero rows past m.
    for (int e = tid; e < META_ROWS * D; e += THREADS) {
        const int r = e / D, i = e % D;
        const __nv_bfloat16 val = r < m ? a.mu[((size_t)h * m + r) * D + i] : __float2bfloat16_rn(0.f);
        *reinterpret_cast<__nv_bfloat16 *>(sm + OFF_MU + (i / 64) * MU_BLOCK + sw128_offset(r, (i % 64) * 2)) = val;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    if (warp < 4) {  // S^T = 0
        uint32_t z[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) z[i] = 0u;
        for (int c = 0; c < D; c += 16) tmem_st16(tmem + tmem_lane(quarter) + T_ST + c, z);
        tmem_wait_st();
    }

    // Every barrier completes one phase per use.  `issued` counts the uses
    // started (TMA or commit, thread 0), `done` the phases this thread has
    // seen complete; the next phase to wait for has parity done & 1.
    enum { B_Q = 0, B_KV = 1, B_SC = 1 + NR, B_Y = 2 + NR, B_ST = 3 + NR };
    uint32_t issued[NBARS], done[NBARS];
#pragma unroll
    for (uint32_t i = 0; i < NBARS; ++i) issued[i] = done[i] = 0;
    auto wait_bar = [&](int b) -> bool {
        const bool ok = mbar_wait(&bars[b], done[b] & 1u, WAIT_LIMIT);
        if (ok) ++done[b];
        return ok;
    };
    auto commit_bar = [&](int b) {
        mma_commit(&bars[b]);
        ++issued[b];
    };
    auto issue_q = [&](int c) {
        mbar_arrive_expect_tx(bar_q, 2 * TILE);
        tma_load_3d(sm + OFF_Q, &tq, bar_q, 0, c * C, unit);
        tma_load_3d(sm + OFF_Q + TILE, &tq, bar_q, 64, c * C, unit);
        ++issued[B_Q];
    };
    auto issue_kv = [&](int c) {
        const int s = c % NR;
        uint8_t *base = sm + OFF_KV + s * KV_SLOT;
        mbar_arrive_expect_tx(&bar_kv[s], 4 * TILE);
        tma_load_3d(base, &tk, &bar_kv[s], 0, c * C, unit);
        tma_load_3d(base + TILE, &tk, &bar_kv[s], 64, c * C, unit);
        tma_load_3d(base + V_OFF, &tv, &bar_kv[s], 0, c * C, unit);
        tma_load_3d(base + V_OFF + TILE, &tv, &bar_kv[s], 64, c * C, unit);
        ++issued[B_KV + s];
    };
    if (tid == 0 && nchunks > 0) {
        issue_q(0);
        issue_kv(0);
        if (nchunks > 1) issue_kv(1);
    }

    // Gate logits of this thread's (key dim, 32 tokens), one chunk ahead.
    const __nv_bfloat16 *gp = a.g + (size_t)unit * L * D + gi;
    float gnext[32];
    auto load_g = [&](int c) {
#pragma unroll
        for (int tt = 0; tt < 32; ++tt) {
            const int tg = c * C + 32 * gth + tt;
            gnext[tt] = tg < L ? __bfloat162float(gp[(size_t)tg * D]) : INFINITY;  // past the end: no decay
        }
    };
    if (nchunks > 0) load_g(0);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    bool aborted = false;
    for (int c = 0; c < nchunks; ++c) {
        const int c0 = c * C, n = min(C, L - c0);
        const uint32_t slot_off = OFF_KV + (c % NR) * KV_SLOT;

        // ---- P1: this chunk's tiles, and the previous state update done ----
        bool ok = wait_bar(B_Q) && wait_bar(B_KV + c % NR);
        if (c > 0) ok = ok && wait_bar(B_ST);
        if (__syncthreads_or(!ok)) { aborted = true; break; }
        tc_fence_after();
        if (tid == 0) {  // window + meta logits
            const uint32_t id64 = instr_desc(64, 64, FMT_BF16, 0, 0), id16 = instr_desc(64, 16, FMT_BF16, 0, 0);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint64_t ad = smem_desc(sb + OFF_Q + (kk / 4) * TILE + (kk % 4) * 32, 16, 1024);
                mma_bf16_ss(tmem + T_SC, ad, smem_desc(sb + OFF_MU + (kk / 4) * MU_BLOCK + (kk % 4) * 32, 16, 1024),
                            id16, kk > 0);
            }
            for (int j = 0; j <= NP; ++j) {
                const int cj = c - NP + j;
                if (cj < 0) continue;
                const uint32_t kb = sb + OFF_KV + (cj % NR) * KV_SLOT;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint64_t ad = smem_desc(sb + OFF_Q + (kk / 4) * TILE + (kk % 4) * 32, 16, 1024);
                    const uint64_t bd = smem_desc(kb + (kk / 4) * TILE + (kk % 4) * 32, 16, 1024);
                    mma_bf16_ss(tmem + T_SC + 16 + 64 * j, ad, bd, id64, kk > 0);
                }
            }
        }

        // ---- P2: log-space gate prefix sums and the folded operands ----
        float b2[32];
        {
            float run = 0.f;
#pragma unroll
            for (int tt = 0; tt < 32; ++tt) {
                run += log2_sigmoid(gnext[tt]);
                b2[tt] = run;
            }
            if (gth == 0) {
                xch[gi] = run;
                first2[gi] = b2[0];
            }
        }
        __syncthreads();
        if (gth == 1) {
            const float off = xch[gi];
#pragma unroll
            for (int tt = 0; tt < 32; ++tt) b2[tt] += off;
        }
#pragma unroll
        for (int tt = 0; tt < 32; ++tt)
            if (32 * gth + tt == n - 1) last2[gi] = b2[tt];
        __syncthreads();
        const float f2 = first2[gi], l2 = last2[gi];
        const float span = f2 - l2;
        const int unsafe = __syncthreads_or(span > SPAN_MAX2);
        if (gth == 0) dec[gi] = ex2(l2);
        if (c + 1 < nchunks) load_g(c + 1);

        float q0[32];
        {
            const float r2 = 0.5f * (f2 + l2);
            const float E = ex2(r2), F = ex2(-0.5f * span);
            const uint32_t blk = (gi / 64) * TILE, byte = (gi % 64) * 2;
#pragma unroll 4
            for (int tt = 0; tt < 32; ++tt) {
                const int t = 32 * gth + tt;
                const uint32_t o = blk + sw128_offset(t, byte);
                const float qv = __bfloat162float(ld_bf16(sm + OFF_Q + o));
                const float kv = __bfloat162float(ld_bf16(sm + slot_off + o));
                float kl;
                if (!unsafe) {
                    const float e = ex2(b2[tt] - r2), ie = ex2(r2 - b2[tt]);
                    const float qr = qv * e, kr = kv * ie;
                    st_bf16(sm + OFF_QZ + o, qr);
                    st_bf16(sm + OFF_KW + o, kr);
                    q0[tt] = qr * E;
                    kl = kr * F;
                } else {
                    reinterpret_cast<float *>(sm + OFF_QZ)[t * D + gi] = b2[tt];
                    q0[tt] = qv * ex2(b2[tt]);
                    kl = kv * ex2(l2 - b2[tt]);
                }
                st_bf16(sm + OFF_KL + o, kl);
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();

        // ---- P3: intra-chunk decayed scores A ----
        if (tid == 0) {
            if (!unsafe) {
                const uint32_t id64 = instr_desc(64, 64, FMT_BF16, 0, 0);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint64_t ad = smem_desc(sb + OFF_QZ + (kk / 4) * TILE + (kk % 4) * 32, 16, 1024);
                    const uint64_t bd = smem_desc(sb + OFF_KW + (kk / 4) * TILE + (kk % 4) * 32, 16, 1024);
                    mma_bf16_ss(tmem + T_A, ad, bd, id64, kk > 0);
                }
            }
            commit_bar(B_SC);
        }
        ok = wait_bar(B_SC);
        if (__syncthreads_or(!ok)) { aborted = true; break; }
        tc_fence_after();
        if (unsafe) {
            // Exact A[t][s] = sum_i q_ti k_si 2^{b2_ti - b2_si}, s <= t, on the CUDA cores.
            // Row t = 16*quarter + (lane & 15); lanes >= 16 take the second 16 of the warp's 32 columns.
            const int t = 16 * quarter + (lane & 15);
            const int s0 = 32 * half + 16 * (lane >> 4);
            const float *bz = reinterpret_cast<const float *>(sm + OFF_QZ);
            float acc[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) acc[e] = 0.f;
            for (int i = 0; i < D; ++i) {
                const uint32_t blk = (i / 64) * TILE, byte = (i % 64) * 2;
                const float qv = __bfloat162float(ld_bf16(sm + OFF_Q + blk + sw128_offset(t, byte)));
                const float bt = bz[t * D + i];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int s = s0 + e;
                    if (s <= t) {
                        const float kv = __bfloat162float(ld_bf16(sm + slot_off + blk + sw128_offset(s, byte)));
                        acc[e] += qv * kv * ex2(bt - bz[s * D + i]);
                    }
                }
            }
            // lanes 16..31 hand their 16 columns to lanes 0..15, which own the TMEM rows
            uint32_t lo[16], hi[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const float other = __shfl_down_sync(0xffffffffu, acc[e], 16);
                lo[e] = __float_as_uint(acc[e]);
                hi[e] = __float_as_uint(other);
            }
            tmem_st16(tmem + tmem_lane(quarter) + T_A + 32 * half, lo);
            tmem_st16(tmem + tmem_lane(quarter) + T_A + 32 * half + 16, hi);
            tmem_wait_st();
            tc_fence_before();
            __syncthreads();
            tc_fence_after();
        }

        // ---- P4: next q tile; q*e^{b} operand; window softmax with sinks -> W ----
        if (tid == 0 && c + 1 < nchunks) {
            fence_proxy_async_smem();
            issue_q(c + 1);
        }
        {
            const uint32_t blk = (gi / 32) * TILE, byte = (gi % 32) * 4;
#pragma unroll
            for (int tt = 0; tt < 32; ++tt)
                *reinterpret_cast<float *>(sm + OFF_QZ + blk + sw128_offset(32 * gth + tt, byte)) = q0[tt];
        }
        {
            const int t = 16 * quarter + (lane & 15);
            const bool own = lane < 16;
            const bool rowok = own && t < n;
            const int tg = c0 + t;
            const int nb = NP + 1;
            const int cbeg = half * 32 * nb, cend = cbeg + 32 * nb;   // this half's band columns
            const int pbase = c0 - 64 * NP;                           // global position of band column 0
            const uint32_t tl = tmem + tmem_lane(quarter);
            float mx = -INFINITY;
            uint32_t r[16];
            if (half == 0) {
                tmem_ld16(tl + T_SC, r);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < META_ROWS; ++j)
                    if (j < m) mx = fmaxf(mx, __uint_as_float(r[j]));
            }
            for (int cc = cbeg; cc < cend; cc += 16) {
                tmem_ld16(tl + T_SC + 16 + cc, r);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int p = pbase + cc + e;
                    if (p >= 0 && p <= tg && p > tg - w) mx = fmaxf(mx, __uint_as_float(r[e]));
                }
            }
            if (own) red[half * 64 + t] = mx;
            __syncthreads();
            const float M = fmaxf(red[t], red[64 + t]);
            const float M2 = M * LOG2E;
            float sum = 0.f;
            if (half == 0) {
                tmem_ld16(tl + T_SC, r);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < META_ROWS; ++j)
                    if (j < m) sum += ex2(__uint_as_float(r[j]) * LOG2E - M2);
            }
            for (int cc = cbeg; cc < cend; cc += 16) {
                tmem_ld16(tl + T_SC + 16 + cc, r);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int p = pbase + cc + e;
                    if (p >= 0 && p <= tg && p > tg - w) sum += ex2(__uint_as_float(r[e]) * LOG2E - M2);
                }
            }
            if (own) red[128 + half * 64 + t] = sum;
            __syncthreads();
            const float inv = a.alpha / (red[128 + t] + red[192 + t]);
            for (int cc = cbeg; cc < cend; cc += 16) {
                tmem_ld16(tl + T_SC + 16 + cc, r);
                uint32_t ra[16];
                const int s0 = cc - 64 * NP;  // column within this chunk (A), when >= 0
                if (s0 >= 0) tmem_ld16(tl + T_A + s0, ra);
                tmem_wait_ld();
                uint32_t packed[8];
#pragma unroll
                for (int e = 0; e < 16; e += 2) {
                    float wv[2];
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int p = pbase + cc + e + u;
                        float x = 0.f;
                        if (p >= 0 && p <= tg && p > tg - w) x = ex2(__uint_as_float(r[e + u]) * LOG2E - M2) * inv;
                        if (s0 >= 0 && p <= tg) x += __uint_as_float(ra[e + u]);
                        wv[u] = rowok ? x : 0.f;
                    }
                    __nv_bfloat162 pr = __floats2bfloat162_rn(wv[0], wv[1]);
                    packed[e / 2] = *reinterpret_cast<uint32_t *>(&pr);
                }
                if (own) {
                    const uint32_t blk = (cc / 64) * TILE, byte = (cc % 64) * 2;
                    *reinterpret_cast<uint4 *>(sm + OFF_KW + blk + sw128_offset(t, byte)) =
                        make_uint4(packed[0], packed[1], packed[2], packed[3]);
                    *reinterpret_cast<uint4 *>(sm + OFF_KW + blk + sw128_offset(t, byte + 16)) =
                        make_uint4(packed[4], packed[5], packed[6], packed[7]);
                }
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();

        // ---- P5: y^T = S^T (q e^{b})^T + V_band^T W^T ----
        if (tid == 0) {
            const uint32_t idt = instr_desc(128, 64, FMT_TF32, 0, 0);
#pragma unroll
            for (int kk = 0; kk < 16; ++kk) {
                const uint64_t bd = smem_desc(sb + OFF_QZ + (kk / 4) * TILE + (kk % 4) * 32, 16, 1024);
                mma_tf32_ts(tmem + T_Y1, tmem + T_ST + kk * 8, bd, idt, kk > 0);
            }
            const uint32_t idv = instr_desc(128, 64, FMT_BF16, 1, 0);
            bool first = true;
            for (int j = 0; j <= NP; ++j) {
                const int cj = c - NP + j;
                if (cj < 0) continue;
                const uint32_t vb = sb + OFF_KV + (cj % NR) * KV_SLOT + V_OFF;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint64_t ad = smem_desc(vb + kk * 2048, 8192, 1024);
                    const uint64_t bd = smem_desc(sb + OFF_KW + j * TILE + kk * 32, 16, 1024);
                    mma_bf16_ss(tmem + T_Y2, ad, bd, idv, first ? 0u : 1u);
                    first = false;
                }
            }
            commit_bar(B_Y);
        }
        ok = wait_bar(B_Y);
        if (__syncthreads_or(!ok)) { aborted = true; break; }
        tc_fence_after();

        // ---- P6: k/v prefetch; decay of S^T; output ----
        if (tid == 0 && c + 2 < nchunks) {
            fence_proxy_async_smem();
            issue_kv(c + 2);
        }
        if (warp < 4) {
            const uint32_t tl = tmem + tmem_lane(quarter) + T_ST;
            for (int cc = 0; cc < D; cc += 16) {
                uint32_t r[16];
                tmem_ld16(tl + cc, r);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 16; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * dec[cc + e]);
                tmem_st16(tl + cc, r);
            }
            tmem_wait_st();
        } else {
            const int j = 32 * quarter + lane;
            __nv_bfloat16 *yp = a.y + ((size_t)unit * L + c0) * D + j;
            for (int cc = 0; cc < C; cc += 16) {
                uint32_t r1[16], r2[16];
                tmem_ld16(tmem + tmem_lane(quarter) + T_Y1 + cc, r1);
                tmem_ld16(tmem + tmem_lane(quarter) + T_Y2 + cc, r2);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    if (cc + e < n) yp[(size_t)(cc + e) * D] = __float2bfloat16_rn(__uint_as_float(r1[e]) + __uint_as_float(r2[e]));
            }
        }
        tc_fence_before();
        __syncthreads();
        tc_fence_after();

        // ---- P7: S^T += V^T (k e^{b_last - b}) ----
        if (tid == 0) {
            const uint32_t ids = instr_desc(128, 128, FMT_BF16, 1, 1);
            const uint32_t vb = sb + slot_off + V_OFF;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_bf16_ss(tmem + T_ST, smem_desc(vb + kk * 2048, 8192, 1024),
                            smem_desc(sb + OFF_KL + kk * 2048, 8192, 1024), ids, 1u);
            commit_bar(B_ST);
        }
    }

    // ---- final state ----
    if (!aborted && nchunks > 0) {
        const bool ok = wait_bar(B_ST);
        if (__syncthreads_or(!ok)) aborted = true;
    }
    tc_fence_after();
    if (aborted) {
        // Record the timeout, then let every copy and product this CTA issued
        // finish (bounded) before tensor memory is released.
        if (tid == 0) {
            atomicExch(&g_device_error, DEV_TIMEOUT);
            for (uint32_t b = 0; b < NBARS; ++b)
                while (done[b] < issued[b] && wait_bar((int)b)) {
                }
        }
    } else if (a.S_out) {
        if (warp < 4) {
            const int j = 32 * quarter + lane;
            float *So = a.S_out + (size_t)unit * D * D + j;
            for (int cc = 0; cc < D; cc += 16) {
                uint32_t r[16];
                tmem_ld16(tmem + tmem_lane(quarter) + T_ST + cc, r);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 16; ++e) So[(size_t)(cc + e) * D] = __uint_as_float(r[e]);
            }
        }
        const int first = max(0, L - w);
        const __nv_bfloat16 *kp = a.k + (size_t)unit * L * D, *vp = a.v + (size_t)unit * L * D;
        __nv_bfloat16 *rk = a.ring_k + (size_t)unit * w * D, *rv = a.ring_v + (size_t)unit * w * D;
        for (int e = tid; e < (L - first) * D; e += THREADS) {
            const int tau = first + e / D, i = e % D;
            rk[(size_t)(tau % w) * D + i] = kp[(size_t)tau * D + i];
            rv[(size_t)(tau % w) * D + i] = vp[(size_t)tau * D + i];
        }
        if (h == 0 && tid == 0) a.pos[unit / a.H] = L;
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, T_COLS);
}

}  // namespace tc
}  // namespace lizard
