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
#include "prefill_cont.cuh"
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
constexpr uint32_t VEC_FLOATS = 4 * 128 + 3 * 128 + 4 * 64;  // xch[4][128], first, last, dec, red[2][2][64]
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
    // Continuation of a sequence (0 / null for a prompt from the empty
    // state): with cont = 1 the CTA takes the start position from pos
    // (take_start_position) and reads the window history, chunks -nprev ..
    // -1, from the ring; S0 [units][D][D] is the start state (may be S_out:
    // the CTA reads it before it writes S_out).
    int cont;
    const float *S0;
    const float *alpha_h;  // per-head anchor weights (null: alpha)
    int group;             // query heads per key/value head (maps tk, tv over B x H / group heads)
    // Sequence segments (a prompt from the empty state only): CTA (unit,
    // seg) covers chunks [seg*seg_chunks, (seg+1)*seg_chunks) and starts
    // from S_init[unit][seg-1] (row = key dim), the state after the earlier
    // segments; its band reaches NP chunks back into the previous segment.
    const float *S_init;
    int seg_chunks, nseg;
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

__device__ __forceinline__ float2 bf2_to_f2(uint32_t u)
{
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u));
}
__device__ __forceinline__ uint32_t f2_to_bf2(float lo, float hi)
{
    __nv_bfloat162 r = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&r);
}

// NP = previous chunks in the window band (ceil((w - 1) / 64)).
template <int NP>
__global__ void __launch_bounds__(THREADS, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                      const __grid_constant__ CUtensorMap tv, const TcArgs a)
{
    constexpr int NB = NP + 1;     // band chunks
    constexpr int PART = 16 * NB;  // band columns per softmax thread (four threads per row)
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = smem_align1024(smem_raw);
    const uint32_t sb = smem_u32(sm);
    float *xch = reinterpret_cast<float *>(sm + OFF_VEC);  // [token quarter 4][128]
    float *first2 = xch + 512, *last2 = first2 + 128, *dec = last2 + 128;
    float *red = dec + 128;  // [pass 2][half 2][row 64]
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + OFF_BAR);
    uint64_t *bar_q = bars, *bar_kv = bars + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + NBARS);
    int64_t *p0_slot = reinterpret_cast<int64_t *>(bars + NBARS + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3, half = warp >> 2;
    const int nseg = a.nseg;
    const int unit = blockIdx.x / nseg, seg = blockIdx.x % nseg, h = unit % a.H;
    const int L = a.L, w = a.w, m = a.m;
    const int nchunks = (L + C - 1) / C;
    const int c_begin = seg * a.seg_chunks, c_end = min(nchunks, c_begin + a.seg_chunks);
    const bool last_seg = seg == nseg - 1;
    // Window history of a continued prompt: NH chunks before the prompt
    // (chunks -NH .. -1), of which tokens -nvalid .. -1 are keys.  A later
    // segment's band starts NP chunks into the previous segment.  Chunk c
    // lives in k/v slot (c - c_begin + NPRE) % NR.
    const int NH = a.cont ? NP : 0;
    const int NPRE = seg > 0 ? NP : NH;
    const int c_lo = c_begin - NPRE;  // first chunk of the first band
    auto slot_of = [&](int c) { return (c - c_lo) % NR; };
    const int kvu = kv_unit(unit, a.H, a.group);  // this head's key/value head
    // Prep mapping: key dims 2ip and 2ip+1, tokens 16*tqr .. 16*tqr+15.
    const int ip = tid & 63, tqr = tid >> 6;
    // Softmax mapping (M = 64 accumulator layout): row srow, column part 2*half + ssub.
    const int srow = 16 * quarter + (lane & 15), ssub = lane >> 4;

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
        *p0_slot = a.cont ? take_start_position(a.pos + unit / a.H, a.H * nseg, L) : 0;
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
    const int64_t p0 = *p0_slot;
    const int nvalid = NH > 0 ? (int)min(p0, (int64_t)(w - 1)) : 0;
    if (NH > 0) {
        // History chunks into slots 0 .. NH-1 (zero rows where no key), in the
        // swizzled layout of a TMA-loaded tile; read from the ring, which this
        // CTA writes only at its end.
        const __nv_bfloat16 *rk = a.ring_k + (size_t)unit * w * D, *rv = a.ring_v + (size_t)unit * w * D;
        const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
        for (int e = tid; e < NH * C * (D / 8); e += THREADS) {
            const int hc = e / (C * (D / 8)), rem = e % (C * (D / 8)), r = rem / (D / 8), i8 = (rem % (D / 8)) * 8;
            const int tau = (hc - NH) * C + r;
            const __nv_bfloat16 *kr = history_row(rk, p0, tau, nvalid, w, D);
            const __nv_bfloat16 *vr = history_row(rv, p0, tau, nvalid, w, D);
            const uint32_t off = hc * KV_SLOT + (i8 / 64) * TILE + sw128_offset(r, (i8 % 64) * 2);
            *reinterpret_cast<uint4 *>(sm + OFF_KV + off) = kr ? *reinterpret_cast<const uint4 *>(kr + i8) : zero;
            *reinterpret_cast<uint4 *>(sm + OFF_KV + V_OFF + off) =
                vr ? *reinterpret_cast<const uint4 *>(vr + i8) : zero;
        }
        fence_proxy_async_smem();
    }
    if (warp < 4) {  // S^T = the state after the earlier segments, or S0 (zero when not given)
        const int j = 32 * quarter + lane;
        const float *Si = seg > 0 ? a.S_init + ((size_t)unit * (nseg - 1) + seg - 1) * D * D + j
                                  : (a.S0 ? a.S0 + (size_t)unit * D * D + j : nullptr);
        for (int c = 0; c < D; c += 16) {
            uint32_t z[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) z[i] = Si ? __float_as_uint(Si[(size_t)(c + i) * D]) : 0u;
            tmem_st16(tmem + tmem_lane(quarter) + T_ST + c, z);
        }
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
        const int s = slot_of(c);
        uint8_t *base = sm + OFF_KV + s * KV_SLOT;
        mbar_arrive_expect_tx(&bar_kv[s], 4 * TILE);
        tma_load_3d(base, &tk, &bar_kv[s], 0, c * C, kvu);
        tma_load_3d(base + TILE, &tk, &bar_kv[s], 64, c * C, kvu);
        tma_load_3d(base + V_OFF, &tv, &bar_kv[s], 0, c * C, kvu);
        tma_load_3d(base + V_OFF + TILE, &tv, &bar_kv[s], 64, c * C, kvu);
        ++issued[B_KV + s];
    };
    if (tid == 0 && c_end > c_begin) {
        if (seg > 0)
            for (int c = c_lo; c < c_begin; ++c) issue_kv(c);  // the previous segment's band chunks
        issue_q(c_begin);
        issue_kv(c_begin);
        if (c_begin + 1 < c_end) issue_kv(c_begin + 1);
    }

    // Gate logits of this thread's two key dims for its 16 tokens, one chunk
    // ahead, as packed bf16 pairs (+inf past the end: no decay).
    const uint32_t *gp = reinterpret_cast<const uint32_t *>(a.g + (size_t)unit * L * D + 2 * ip);
    uint32_t gnext[16];
    auto load_g = [&](int c) {
#pragma unroll
        for (int tt = 0; tt < 16; ++tt) {
            const int tg = c * C + 16 * tqr + tt;
            gnext[tt] = tg < L ? gp[(size_t)tg * (D / 2)] : 0x7F807F80u;
        }
    };
    if (c_end > c_begin) load_g(c_begin);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    bool aborted = false;
    for (int c = c_begin; c < c_end; ++c) {
        const int c0 = c * C, n = min(C, L - c0);
        const uint32_t slot_off = OFF_KV + slot_of(c) * KV_SLOT;

        // ---- P1: this chunk's tiles, and the previous state update done ----
        bool ok = wait_bar(B_Q) && wait_bar(B_KV + slot_of(c));
        if (c == c_begin && seg > 0)
            for (int cp = c_lo; cp < c_begin; ++cp) ok = ok && wait_bar(B_KV + slot_of(cp));
        if (c > c_begin) ok = ok && wait_bar(B_ST);
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
#pragma unroll
            for (int j = 0; j <= NP; ++j) {
                const int cj = c - NP + j;
                if (cj < c_lo) continue;
                const uint32_t kb = sb + OFF_KV + slot_of(cj) * KV_SLOT;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint64_t ad = smem_desc(sb + OFF_Q + (kk / 4) * TILE + (kk % 4) * 32, 16, 1024);
                    const uint64_t bd = smem_desc(kb + (kk / 4) * TILE + (kk % 4) * 32, 16, 1024);
                    mma_bf16_ss(tmem + T_SC + 16 + 64 * j, ad, bd, id64, kk > 0);
                }
            }
        }

        // ---- P2: log-space gate prefix sums and the folded operands ----
        float b2a[16], b2b[16];
        {
            float ra = 0.f, rb = 0.f;
#pragma unroll
            for (int tt = 0; tt < 16; ++tt) {
                const float2 gg = bf2_to_f2(gnext[tt]);
                ra += log2_sigmoid(gg.x);
                rb += log2_sigmoid(gg.y);
                b2a[tt] = ra;
                b2b[tt] = rb;
            }
            xch[tqr * 128 + 2 * ip] = ra;
            xch[tqr * 128 + 2 * ip + 1] = rb;
            if (tqr == 0) {
                first2[2 * ip] = b2a[0];
                first2[2 * ip + 1] = b2b[0];
            }
        }
        __syncthreads();
        {
            float oa = 0.f, ob = 0.f;
            for (int qq = 0; qq < tqr; ++qq) {
                oa += xch[qq * 128 + 2 * ip];
                ob += xch[qq * 128 + 2 * ip + 1];
            }
#pragma unroll
            for (int tt = 0; tt < 16; ++tt) {
                b2a[tt] += oa;
                b2b[tt] += ob;
                if (16 * tqr + tt == n - 1) {
                    last2[2 * ip] = b2a[tt];
                    last2[2 * ip + 1] = b2b[tt];
                }
            }
        }
        __syncthreads();
        const float f2a = first2[2 * ip], l2a = last2[2 * ip];
        const float f2b = first2[2 * ip + 1], l2b = last2[2 * ip + 1];
        const int unsafe = __syncthreads_or(f2a - l2a > SPAN_MAX2 || f2b - l2b > SPAN_MAX2);
        if (tqr == 0) {
            dec[2 * ip] = ex2(l2a);
            dec[2 * ip + 1] = ex2(l2b);
        }
        if (c + 1 < c_end) load_g(c + 1);

        float q0a[16], q0b[16];
        {
            const float r2a = 0.5f * (f2a + l2a), r2b = 0.5f * (f2b + l2b);
            const float Ea = ex2(r2a), Eb = ex2(r2b);
            const float Fa = ex2(0.5f * (l2a - f2a)), Fb = ex2(0.5f * (l2b - f2b));
            const uint32_t blk = (ip / 32) * TILE, byte = (ip % 32) * 4;
#pragma unroll
            for (int tt = 0; tt < 16; ++tt) {
                const int t = 16 * tqr + tt;
                const uint32_t o = blk + sw128_offset(t, byte);
                const float2 qv = bf2_to_f2(*reinterpret_cast<const uint32_t *>(sm + OFF_Q + o));
                const float2 kv = bf2_to_f2(*reinterpret_cast<const uint32_t *>(sm + slot_off + o));
                float kla, klb;
                if (!unsafe) {
                    const float qra = qv.x * ex2(b2a[tt] - r2a), qrb = qv.y * ex2(b2b[tt] - r2b);
                    const float kra = kv.x * ex2(r2a - b2a[tt]), krb = kv.y * ex2(r2b - b2b[tt]);
                    *reinterpret_cast<uint32_t *>(sm + OFF_QZ + o) = f2_to_bf2(qra, qrb);
                    *reinterpret_cast<uint32_t *>(sm + OFF_KW + o) = f2_to_bf2(kra, krb);
                    q0a[tt] = qra * Ea;
                    q0b[tt] = qrb * Eb;
                    kla = kra * Fa;
                    klb = krb * Fb;
                } else {
                    *reinterpret_cast<float2 *>(sm + OFF_QZ + ((size_t)t * D + 2 * ip) * 4) = make_float2(b2a[tt], b2b[tt]);
                    q0a[tt] = qv.x * ex2(b2a[tt]);
                    q0b[tt] = qv.y * ex2(b2b[tt]);
                    kla = kv.x * ex2(l2a - b2a[tt]);
                    klb = kv.y * ex2(l2b - b2b[tt]);
                }
                *reinterpret_cast<uint32_t *>(sm + OFF_KL + o) = f2_to_bf2(kla, klb);
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
            // Exact A[t][s] = sum_i q_ti k_si 2^{b2_ti - b2_si} for s <= t on
            // the CUDA cores; this thread's row srow, columns 16p .. 16p+15.
            const int t = srow, s0 = 16 * (2 * half + ssub);
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
            uint32_t r[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) r[e] = __float_as_uint(acc[e]);
            tmem_st16_x2<16>(tmem + tmem_lane(quarter) + T_A + 32 * half, r);
            tmem_wait_st();
            tc_fence_before();
            __syncthreads();
            tc_fence_after();
        }

        // ---- P4: next q tile; q*e^{b} operand and y^T part 1; softmax -> W ----
        if (tid == 0 && c + 1 < c_end) {
            fence_proxy_async_smem();
            issue_q(c + 1);
        }
        {
            const uint32_t blk = (ip / 16) * TILE, byte = (ip % 16) * 8;
#pragma unroll
            for (int tt = 0; tt < 16; ++tt)
                *reinterpret_cast<float2 *>(sm + OFF_QZ + blk + sw128_offset(16 * tqr + tt, byte)) =
                    make_float2(q0a[tt], q0b[tt]);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (tid == 0) {  // y^T part 1 = S^T (q e^{b})^T, overlapping the softmax below
            const uint32_t idt = instr_desc(128, 64, FMT_TF32, 0, 0);
#pragma unroll
            for (int kk = 0; kk < 16; ++kk) {
                const uint64_t bd = smem_desc(sb + OFF_QZ + (kk / 4) * TILE + (kk % 4) * 32, 16, 1024);
                mma_tf32_ts(tmem + T_Y1, tmem + T_ST + kk * 8, bd, idt, kk > 0);
            }
        }
        {
            const int t = srow, tg = c0 + t, p = 2 * half + ssub;
            const bool rowok = t < n;
            const int pbase = c0 - 64 * NP;  // global position of band column 0
            const uint32_t tl = tmem + tmem_lane(quarter);
            uint32_t rr[NB][16], rm[16];
#pragma unroll
            for (int gq = 0; gq < NB; ++gq) tmem_ld16_x2<PART>(tl + T_SC + 16 + 2 * PART * half + 16 * gq, rr[gq]);
            tmem_ld16_x2<PART>(tl + T_SC, rm);
            tmem_wait_ld();
            const bool meta_owner = half == 0 && ssub == 0;
            float x[PART];
            float mx = -INFINITY;
#pragma unroll
            for (int gq = 0; gq < NB; ++gq)
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int pp = pbase + PART * p + 16 * gq + e;
                    const bool valid = pp >= -nvalid && pp <= tg && pp > tg - w;
                    x[16 * gq + e] = valid ? __uint_as_float(rr[gq][e]) : -INFINITY;
                    mx = fmaxf(mx, x[16 * gq + e]);
                }
            if (meta_owner) {
#pragma unroll
                for (int j = 0; j < META_ROWS; ++j)
                    if (j < m) mx = fmaxf(mx, __uint_as_float(rm[j]));
            }
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
            if (ssub == 0) red[half * 64 + t] = mx;
            __syncthreads();
            const float M2 = fmaxf(red[t], red[64 + t]) * LOG2E;
            float sum = 0.f;
#pragma unroll
            for (int k = 0; k < PART; ++k) {
                x[k] = ex2(x[k] * LOG2E - M2);
                sum += x[k];
            }
            if (meta_owner) {
#pragma unroll
                for (int j = 0; j < META_ROWS; ++j)
                    if (j < m) sum += ex2(__uint_as_float(rm[j]) * LOG2E - M2);
            }
            sum += __shfl_xor_sync(0xffffffffu, sum, 16);
            if (ssub == 0) red[128 + half * 64 + t] = sum;
            __syncthreads();
            const float inv = head_alpha(a.alpha_h, a.alpha, h) / (red[128 + t] + red[192 + t]);
#pragma unroll
            for (int gq = 0; gq < NB; ++gq) {
                const int colw = 2 * PART * half + 16 * gq;  // band column of lanes 0..15 (lanes 16..31: + PART)
                const int col0 = colw + PART * ssub;         // this thread's 16 band columns start here
                uint32_t ra[16];
                const bool need_a = colw + PART + 16 > 64 * NP;  // some lane reaches the current chunk
                if (need_a) {
                    tmem_ld16_x2<PART>(tl + T_A + colw - 64 * NP, ra);
                    tmem_wait_ld();
                }
                uint32_t packed[8];
#pragma unroll
                for (int e = 0; e < 16; e += 2) {
                    float wv[2];
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int col = col0 + e + u, s = col - 64 * NP;
                        float v = x[16 * gq + e + u] * inv;
                        if (need_a && s >= 0 && pbase + col <= tg) v += __uint_as_float(ra[e + u]);
                        wv[u] = rowok ? v : 0.f;
                    }
                    packed[e / 2] = f2_to_bf2(wv[0], wv[1]);
                }
                const uint32_t blk = (col0 / 64) * TILE, byte = (col0 % 64) * 2;
                *reinterpret_cast<uint4 *>(sm + OFF_KW + blk + sw128_offset(t, byte)) =
                    make_uint4(packed[0], packed[1], packed[2], packed[3]);
                *reinterpret_cast<uint4 *>(sm + OFF_KW + blk + sw128_offset(t, byte + 16)) =
                    make_uint4(packed[4], packed[5], packed[6], packed[7]);
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();

        // ---- P5: y^T part 2 = V_band^T W^T ----
        if (tid == 0) {
            const uint32_t idv = instr_desc(128, 64, FMT_BF16, 1, 0);
            bool first = true;
#pragma unroll
            for (int j = 0; j <= NP; ++j) {
                const int cj = c - NP + j;
                if (cj < c_lo) continue;
                const uint32_t vb = sb + OFF_KV + slot_of(cj) * KV_SLOT + V_OFF;
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
        if (tid == 0 && c + 2 < c_end) {
            fence_proxy_async_smem();
            issue_kv(c + 2);
        }
        if (warp < 4) {
            const uint32_t tl = tmem + tmem_lane(quarter) + T_ST;
#pragma unroll
            for (int cc = 0; cc < D; cc += 32) {
                uint32_t r0[16], r1[16];
                tmem_ld16(tl + cc, r0);
                tmem_ld16(tl + cc + 16, r1);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    r0[e] = __float_as_uint(__uint_as_float(r0[e]) * dec[cc + e]);
                    r1[e] = __float_as_uint(__uint_as_float(r1[e]) * dec[cc + 16 + e]);
                }
                tmem_st16(tl + cc, r0);
                tmem_st16(tl + cc + 16, r1);
            }
            tmem_wait_st();
        } else {
            const int j = 32 * quarter + lane;
            __nv_bfloat16 *yp = a.y + ((size_t)unit * L + c0) * D + j;
#pragma unroll
            for (int cc = 0; cc < C; cc += 16) {
                uint32_t r1[16], r2[16];
                tmem_ld16(tmem + tmem_lane(quarter) + T_Y1 + cc, r1);
                tmem_ld16(tmem + tmem_lane(quarter) + T_Y2 + cc, r2);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    if (cc + e < n)
                        yp[(size_t)(cc + e) * D] = __float2bfloat16_rn(__uint_as_float(r1[e]) + __uint_as_float(r2[e]));
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
    if (!aborted && c_end > c_begin) {
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
    } else if (a.S_out && last_seg) {
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
        const __nv_bfloat16 *kp = a.k + (size_t)kvu * L * D, *vp = a.v + (size_t)kvu * L * D;
        __nv_bfloat16 *rk = a.ring_k + (size_t)unit * w * D, *rv = a.ring_v + (size_t)unit * w * D;
        for (int e = tid; e < (L - first) * D; e += THREADS) {
            const int tau = first + e / D, i = e % D;
            const size_t slot = (size_t)((p0 + tau) % w);  // token p0 + tau
            rk[slot * D + i] = kp[(size_t)tau * D + i];
            rv[slot * D + i] = vp[(size_t)tau * D + i];
        }
        if (!a.cont && h == 0 && tid == 0) a.pos[unit / a.H] = L;  // (a continued prompt advanced pos at its start)
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, T_COLS);
}

}  // namespace tc
}  // namespace lizard
