// prefill_state.cuh -- segment end states of the gated linear attention
// branch, for prefills split into sequence segments (bf16, d = 128).
//
// Lizard (gist.science/de) section 2 item 1: the state follows
// S_t = diag(sigmoid(g_t)) S_{t-1} + k_t^T v_t.  Unrolled over a segment
// [t0, t1) that starts from S = 0:
//
//   dS = sum_{t0<=s<t1} diag(2^{suf_s}) k_s^T v_s,   suf_s = sum_{s<r<t1} log2 sigmoid(g_r)
//   Lam = sum_{t0<=r<t1} log2 sigmoid(g_r)            (the segment's total decay, per key dim)
//
// so that S_end = diag(2^Lam) S_start + dS.  Every exponent suf_s is <= 0,
// so no rescaling of the accumulator is needed: the chunks are walked from
// the end of the segment backwards and each chunk's k is scaled by 2^{suf}
// (the log-space fold of the gate into the key operand, as in the page's
// "Hardware-bewusster Algorithmus" section) and accumulated with one
// tensor-core product per chunk: dS^T += V^T (k 2^{suf}).
//
// Roles (14 warps): warp 0 TMA (g, k, v tiles, two stages), warp 1 MMA
// issuer, warps 2-5 zero the accumulator and write dS at the end, warps
// 6-13 gate prep (log-sigmoid, suffix sums, the scaled key tile).  Waits
// are bounded as in the prefill kernel.
#pragma once

#include "common.cuh"
#include "sm100.cuh"
#include "prefill_ws.cuh"

namespace lizard {
namespace seg {

using namespace sm100;
using ws::C;
using ws::D;
using ws::KB_T;

constexpr int NWARPS = 14;
constexpr int THREADS = NWARPS * 32;
constexpr int W_TMA = 0, W_MMA = 1, W_OUT = 2, W_PREP = 6;
constexpr int OUT_N = 128, PREP_N = 256;
enum : int { NB_OUT_R = 1, NB_PREP = 2, NB_PREP_R = 3 };
constexpr int ST = 2;  // stages

// Shared memory: per stage g | k | v (16 KiB each), then one scaled-key
// tile per stage.
constexpr uint32_t STAGE = 3 * 2 * KB_T;
constexpr uint32_t OFF_KH = ST * STAGE;
constexpr uint32_t OFF_TOT = OFF_KH + ST * 2 * KB_T;  // [4][128] fp32 quarter totals
constexpr uint32_t OFF_BAR = OFF_TOT + 4 * 128 * 4;
constexpr int NBAR = 4 * ST + 2;
constexpr uint32_t OFF_FLAG = OFF_BAR + NBAR * 8;
constexpr uint32_t OFF_TSLOT = OFF_FLAG + 16;
constexpr uint32_t SMEM_BYTES = OFF_TSLOT + 16 + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

// Every segment but the last is walked as nsub sub-blocks of sub_chunks
// chunks (the walk is latency-bound: more, shorter walks side by side).
struct SegArgs {
    float *dS;      // [units][(nseg-1) nsub][D][D] fp32, row = key dim
    float *lam;     // [units][(nseg-1) nsub][D] fp32 (base-2 log of the sub-block's decay)
    int L, seg_chunks, nseg;
    int H, group;   // query heads per key/value head (tk, tv map B x H / group heads)
    int nsub, sub_chunks;
};

// grid = units * (nseg - 1) * nsub: CTA (unit, q), q = p nsub + b, covers
// sub-block b of segment p: chunks [p seg_chunks + b sub_chunks, ...), at
// most sub_chunks of them and none past the segment.
__global__ void __launch_bounds__(THREADS, 1)
    segment_state_kernel(const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                         const __grid_constant__ CUtensorMap tg, const SegArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = smem_align1024(smem_raw);
    const uint32_t sb = smem_u32(sm);
    float *tot = reinterpret_cast<float *>(sm + OFF_TOT);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + OFF_BAR);
    uint64_t *full = bars, *empty = bars + ST, *kh_full = bars + 2 * ST, *kh_free = bars + 3 * ST;
    uint64_t *drain = bars + 4 * ST, *done = drain + 1;
    volatile int *abort_f = reinterpret_cast<volatile int *>(sm + OFF_FLAG);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + OFF_TSLOT);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nsp = (a.nseg - 1) * a.nsub;  // sub-blocks per unit
    const int unit = blockIdx.x / nsp, p = blockIdx.x % nsp;
    const int seg = p / a.nsub, sb_i = p % a.nsub;
    const int nchunks_all = (a.L + C - 1) / C;
    const int seg_end = min(nchunks_all, (seg + 1) * a.seg_chunks);
    const int c_begin = seg * a.seg_chunks + sb_i * a.sub_chunks, c_end = min(seg_end, c_begin + a.sub_chunks);
    const int nch = max(0, c_end - c_begin);

    if (warp == W_MMA) {
        tmem_alloc(tmem_slot, 128);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int i = 0; i < ST; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 2);   // prep done with g, k; the product done with v
            mbar_init(&kh_full[i], 1);
            mbar_init(&kh_free[i], 1);
        }
        mbar_init(drain, 1);
        mbar_init(done, 1);
        *abort_f = 0;
        fence_mbar_init();
        prefetch_tmap(&tk);
        prefetch_tmap(&tv);
        prefetch_tmap(&tg);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    bool failed = false;
    auto give_up = [&]() {
        failed = true;
        *abort_f = 1;
        atomicExch(&g_device_error, DEV_TIMEOUT);
    };

    if (warp == W_TMA) {
        if (lane == 0) {
            uint32_t issued[ST] = {};
            // the segment's chunks, last first
            for (int i = 0; i < nch; ++i) {
                const int c = c_end - 1 - i, s = i % ST;
                if (i >= ST && !ws::bwait(&empty[s], i / ST - 1, abort_f)) { give_up(); break; }
                uint8_t *base = sm + s * STAGE;
                mbar_arrive_expect_tx(&full[s], 3 * 2 * KB_T);
                tma_load_3d(base, &tg, &full[s], 0, c * C, unit);
                tma_load_3d(base + KB_T, &tg, &full[s], 64, c * C, unit);
                tma_load_3d(base + 2 * KB_T, &tk, &full[s], 0, c * C, kv_unit(unit, a.H, a.group));
                tma_load_3d(base + 3 * KB_T, &tk, &full[s], 64, c * C, kv_unit(unit, a.H, a.group));
                tma_load_3d(base + 4 * KB_T, &tv, &full[s], 0, c * C, kv_unit(unit, a.H, a.group));
                tma_load_3d(base + 5 * KB_T, &tv, &full[s], 64, c * C, kv_unit(unit, a.H, a.group));
                ++issued[s];
            }
            for (int s = 0; s < ST; ++s)
                if (issued[s]) ws::bwait(&full[s], issued[s] - 1, abort_f);
        }
        __syncwarp();
    } else if (warp == W_MMA) {
        if (lane == 0) {
            const uint32_t id_st = instr_desc(128, 128, FMT_BF16, 1, 1);
            for (int i = 0; i < nch; ++i) {
                const int s = i % ST;
                if (!ws::bwait(&full[s], i / ST, abort_f) || !ws::bwait(&kh_full[s], i / ST, abort_f)) {
                    give_up();
                    break;
                }
                tc_fence_after();
                const uint32_t vb = sb + s * STAGE + 4 * KB_T, kb = sb + OFF_KH + s * 2 * KB_T;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16_ss(tmem, smem_desc(vb + kk * 2048, KB_T, 1024), smem_desc(kb + kk * 2048, KB_T, 1024),
                                id_st, (i > 0 || kk > 0) ? 1u : 0u);
                mma_commit(&empty[s]);
                mma_commit(&kh_free[s]);
            }
            mma_commit(done);
            ws::bwait(done, 0, abort_f);
        }
        __syncwarp();
    } else if (warp >= W_OUT && warp < W_OUT + 4) {
        // Zero the accumulator (an empty segment still writes dS = 0), wait
        // for the last product, write dS^T[j][i] -> dS[i][j].
        const int quarter = warp & 3, j = 32 * quarter + lane;
        const uint32_t tl = tmem + ((32u * quarter) << 16);
        if (nch == 0) {
            uint32_t z[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) z[e] = 0u;
            for (int cc = 0; cc < D; cc += 16) tmem_st16(tl + cc, z);
            tmem_wait_st();
        }
        const bool ok = ws::role_wait(warp == W_OUT, lane, NB_OUT_R, OUT_N,
                                      [&] { return nch == 0 || ws::bwait(done, 0, abort_f); });
        if (ok) {
            tc_fence_after();
            float *dst = a.dS + ((size_t)unit * nsp + p) * D * D + j;
#pragma unroll 1
            for (int cc = 0; cc < D; cc += 16) {
                uint32_t r[16];
                tmem_ld16(tl + cc, r);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 16; ++e) dst[(size_t)(cc + e) * D] = __uint_as_float(r[e]);
            }
        } else {
            give_up();
        }
    } else if (warp >= W_PREP && warp < W_PREP + 8) {
        const int tp = tid - W_PREP * 32;
        const int pr = tp & 63, hq = tp >> 6;     // key dims 2pr, 2pr+1; tokens 16 hq .. 16 hq + 15
        const uint32_t kblk = pr / 32, kbyte = (pr % 32) * 4;
        float2 off = make_float2(0.f, 0.f);       // sum of log-gates of the later chunks of the segment
        for (int i = 0; i < nch; ++i) {
            const int c = c_end - 1 - i, s = i % ST;
            const int n = min(C, a.L - c * C);
            if (!ws::role_wait(warp == W_PREP, lane, NB_PREP_R, PREP_N, [&] {
                    return ws::bwait(&full[s], i / ST, abort_f) && (i < ST || ws::bwait(&kh_free[s], i / ST - 1, abort_f));
                })) { give_up(); break; }
            const uint8_t *gt = sm + s * STAGE + kblk * KB_T, *kt = sm + s * STAGE + 2 * KB_T + kblk * KB_T;
            float2 cs[16];
            float2 run = make_float2(0.f, 0.f);
#pragma unroll
            for (int tt = 0; tt < 16; ++tt) {
                const int t = 16 * hq + tt;
                const float2 l = ws::log2_sigmoid2(ws::bf2_to_f2(*reinterpret_cast<const uint32_t *>(gt + sw128_offset(t, kbyte))));
                if (t < n) run = ws::add2(run, l);
                cs[tt] = run;
            }
            tot[hq * 128 + 2 * pr] = run.x;
            tot[hq * 128 + 2 * pr + 1] = run.y;
            asm volatile("bar.sync %0, %1;" ::"r"((int)NB_PREP), "r"(PREP_N) : "memory");
            float2 pre = make_float2(0.f, 0.f), total = make_float2(0.f, 0.f);
#pragma unroll
            for (int qq = 0; qq < 4; ++qq) {
                const float2 T = make_float2(tot[qq * 128 + 2 * pr], tot[qq * 128 + 2 * pr + 1]);
                if (qq < hq) pre = ws::add2(pre, T);
                total = ws::add2(total, T);
            }
            // suffix of token t within the segment: (total - (pre + cs_t)) + off <= 0
            const float2 base = make_float2(total.x - pre.x + off.x, total.y - pre.y + off.y);
            uint8_t *kh = sm + OFF_KH + s * 2 * KB_T + kblk * KB_T;
#pragma unroll
            for (int tt = 0; tt < 16; ++tt) {
                const uint32_t o = sw128_offset(16 * hq + tt, kbyte);
                const float2 kv = ws::bf2_to_f2(*reinterpret_cast<const uint32_t *>(kt + o));
                const float2 e = make_float2(base.x - cs[tt].x, base.y - cs[tt].y);
                const float2 kk = ws::mul2(kv, make_float2(ws::ex2(e.x), ws::ex2(e.y)));
                *reinterpret_cast<uint32_t *>(kh + o) = ws::f2_to_bf2(kk.x, kk.y);
            }
            off = ws::add2(off, total);
            fence_proxy_async_smem();
            asm volatile("bar.sync %0, %1;" ::"r"((int)NB_PREP), "r"(PREP_N) : "memory");
            if (tp == 0) {
                mbar_arrive(&kh_full[s]);
                mbar_arrive(&empty[s]);
            }
        }
        if (!failed && hq == 0) {
            float *lam = a.lam + ((size_t)unit * nsp + p) * D;
            lam[2 * pr] = off.x;
            lam[2 * pr + 1] = off.y;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == W_MMA) tmem_dealloc(tmem, 128);
}

// A continued prompt (Lizard, gist.science/de section 2 items 1-2: the
// state and the anchor window carry on from earlier tokens): its start
// state S0 and the state's pos and ring, from which the scan copies what the
// first segment reads -- the last segment writes S and the ring in place.
// All null for a prompt from the empty state.
struct ScanCont {
    const float *S0;
    float *S0_copy;                          // [units][D][D]
    const __nv_bfloat16 *ring_k, *ring_v;    // [units][w][D]
    const int64_t *pos;                      // [B]
    __nv_bfloat16 *hist;                     // [units][2][C][D]: keys, values of tokens -C .. -1
    int H, w;
};

// Segment start states: S_start(0) = S0 (zero when S0 is null), the state
// folded through the sub-blocks in order, S <- diag(2^{Lam_q}) S + dS_q, and
// after the last sub-block of segment p written to Sst[u][p] = S_start(p + 1)
// (Sst may be dS itself when nsub = 1: each element is read before it is
// written, by the same thread).  For a continued prompt
// the first segment's inputs are copied as well: S0, and the window history
// (row r = token r - C, from ring slot (p0 + r - C) % w with p0 = the low 40
// bits of pos, as the prefill takes it; zero rows where no key).  One
// thread per state element and unit.
__global__ void segment_scan_kernel(float *dS, const float *lam, float *Sst, int units, int nseg, int nsub,
                                    ScanCont sc)
{
    const int nsp = nseg - 1, nq = nsp * nsub;
    const int u = blockIdx.y;
    const int e = blockIdx.x * blockDim.x + threadIdx.x;  // i * D + j
    if (u >= units || e >= D * D) return;
    if (sc.hist && e < 2 * C * (D / 8)) {
        const int kv = e / (C * (D / 8)), r = (e / (D / 8)) % C, i8 = (e % (D / 8)) * 8;
        const int64_t p0 = (int64_t)((unsigned long long)sc.pos[u / sc.H] & (CONT_POS_TICK - 1));
        const int nvalid = (int)min(p0, (int64_t)(sc.w - 1));
        const __nv_bfloat16 *ring = (kv ? sc.ring_v : sc.ring_k) + (size_t)u * sc.w * D;
        uint4 val = make_uint4(0u, 0u, 0u, 0u);
        if (r - C >= -nvalid)
            val = *reinterpret_cast<const uint4 *>(ring + (size_t)((p0 + r - C) % sc.w) * D + i8);
        *reinterpret_cast<uint4 *>(sc.hist + (((size_t)u * 2 + kv) * C + r) * D + i8) = val;
    }
    const int i = e / D;
    float S = sc.S0 ? sc.S0[(size_t)u * D * D + e] : 0.f;
    if (sc.S0_copy) sc.S0_copy[(size_t)u * D * D + e] = S;
    for (int q = 0; q < nq; ++q) {
        const size_t off = ((size_t)u * nq + q) * D * D + e;
        S = exp2f(lam[((size_t)u * nq + q) * D + i]) * S + dS[off];
        if ((q + 1) % nsub == 0) Sst[((size_t)u * nsp + q / nsub) * D * D + e] = S;
    }
}

}  // namespace seg
}  // namespace lizard
