// prefill_simt.cuh -- chunked prefill of the Lizard operator on CUDA cores.
//
// Exact fp32 chunkwise form of the gated linear attention recurrence
// (Lizard, gist.science/de section 2 item 1) with the anchor window and
// meta-memory sinks (item 2) and the alpha combine (item 3).
//
// Chunk c covers tokens c0 .. c0+C-1.  With b_t = sum_{r=c0..t} log sigmoid(g_r)
// (per key dim, fp32, log space as in the "Hardware-bewusster Algorithmus"
// section of the same page):
//   y_t   = (q_t * e^{b_t}) S_{c-1}                                 inter-chunk
//         + sum_{c0<=s<=t} (sum_i q_ti k_si e^{b_ti - b_si}) v_s    intra-chunk
//         + alpha * ya_t                                            anchor
//   S_c   = diag(e^{b_last}) S_{c-1} + sum_s (k_s * e^{b_last - b_s})^T v_s
// Every exponent above is <= 0, so nothing overflows for any gate values.
// One CTA per (batch, head) walks the chunks in order with S in shared
// memory; at d = 256 the value dims are split over four CTAs (64 each, the
// columns of S, y and the anchor sum are independent; each CTA scores the
// whole window) and the chunks are 32 tokens, so that S's slice and the
// chunk tiles fit.  This kernel has no tensor-core path; it is the exact
// CUDA-core formulation of the chunked algorithm.
#pragma once

#include "common.cuh"
#include "prefill_cont.cuh"

namespace lizard {

struct PrefillArgs {
    const void *q, *k, *v, *g, *mu;
    void *y;
    float alpha;
    int B, H, L, w, m;
    // optional state out
    float *S_out;
    void *ring_k, *ring_v;
    int64_t *pos;
    // Continuation of a sequence (0 / null for a prompt from the empty
    // state): with cont = 1 every CTA takes the start position from pos
    // (take_start_position) and reads the window history from the ring; S0
    // [units][d][d] is the start state (may be S_out: each CTA reads its own
    // unit's S0 before it writes S_out).
    int cont;
    const float *S0;
    // Variants: per-head anchor weights alpha_h[H] (null: alpha for every
    // head) and grouped key/value heads (k, v hold B x H / group heads).
    const float *alpha_h;
    int group;
};

constexpr int SIMT_THREADS = 256;
constexpr int SIMT_WARPS = SIMT_THREADS / 32;

// Chunk length, value dims per CTA and CTAs per (batch, head) for head dim D.
template <int D>
struct SimtShape {
    static constexpr int C = D > 128 ? 32 : 64;
    static constexpr int DV = D > 128 ? 64 : D;
    static constexpr int NSL = D / DV;
    static_assert(D % DV == 0 && DV % 32 == 0, "value slices of whole warps");
};

template <int D>
size_t prefill_simt_smem_bytes(int w, int m)
{
    using SS = SimtShape<D>;
    const int LD = D + 1;
    return sizeof(float) * ((size_t)D * SS::DV + 3 * (size_t)SS::C * LD + (size_t)SS::C * SS::DV +
                            (size_t)SS::C * SS::C + (size_t)SIMT_WARPS * (w + m));
}

// grid = NSL * B * H; CTA (unit, slice) owns value columns j0 .. j0 + DV - 1.
template <typename T, int D>
__global__ void __launch_bounds__(SIMT_THREADS, 1) prefill_simt_kernel(PrefillArgs a)
{
    using SS = SimtShape<D>;
    constexpr int C = SS::C, DV = SS::DV, NSL = SS::NSL;
    constexpr int LD = D + 1;       // padded row stride (column reads stay bank-conflict free)
    constexpr int JPL = DV / 32;    // output columns per lane
    const int unit = blockIdx.x / NSL, slice = blockIdx.x % NSL, j0 = slice * DV, h = unit % a.H;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int L = a.L, w = a.w, m = a.m;

    extern __shared__ float sm[];
    float *S_s = sm;                       // [D][DV]  (key dim i, this CTA's value dims)
    float *q_s = S_s + D * DV;             // [C][LD]
    float *k_s = q_s + C * LD;             // [C][LD]  (becomes k * e^{b_last - b})
    float *b_s = k_s + C * LD;             // [C][LD]  cumulative log gate
    float *v_s = b_s + C * LD;             // [C][DV]
    float *A_s = v_s + C * DV;             // [C][C]
    float *sc_all = A_s + C * C;           // [warps][w + m]
    float *sc = sc_all + warp * (w + m);

    const size_t base = (size_t)unit * L * D;
    const T *q = static_cast<const T *>(a.q) + base;
    const size_t kvbase = (size_t)kv_unit(unit, a.H, a.group) * L * D;
    const T *k = static_cast<const T *>(a.k) + kvbase;
    const T *v = static_cast<const T *>(a.v) + kvbase;
    const T *g = static_cast<const T *>(a.g) + base;
    const T *mu = static_cast<const T *>(a.mu) + (size_t)h * m * D;
    T *y = static_cast<T *>(a.y) + base;
    // Start position p0 (0 for a prompt from the empty state) and the
    // window keys before the prompt: tokens -nvalid .. -1, ring slot (p0 + tau) % w.
    __shared__ int64_t p0_sh;
    if (tid == 0) p0_sh = a.cont ? take_start_position(a.pos + unit / a.H, a.H * NSL, L) : 0;
    const T *ring_k = a.cont ? static_cast<const T *>(a.ring_k) + (size_t)unit * w * D : nullptr;
    const T *ring_v = a.cont ? static_cast<const T *>(a.ring_v) + (size_t)unit * w * D : nullptr;

    const float *S0 = a.S0 ? a.S0 + (size_t)unit * D * D : nullptr;
    for (int e = tid; e < D * DV; e += SIMT_THREADS) S_s[e] = S0 ? S0[(e / DV) * D + j0 + e % DV] : 0.f;
    __syncthreads();
    const int64_t p0 = p0_sh;
    const int nvalid = a.cont ? (int)min(p0, (int64_t)(w - 1)) : 0;

    for (int c0 = 0; c0 < L; c0 += C) {
        const int n = min(C, L - c0);
        __syncthreads();
        // 1. Chunk tiles (rows >= n are zero: no key, no value, no decay).
        for (int e = tid; e < C * D; e += SIMT_THREADS) {
            const int t = e / D, i = e % D;
            const bool ok = t < n;
            const size_t off = (size_t)(c0 + t) * D + i;
            q_s[t * LD + i] = ok ? to_f32(q[off]) : 0.f;
            k_s[t * LD + i] = ok ? to_f32(k[off]) : 0.f;
            b_s[t * LD + i] = ok ? log_sigmoid(to_f32(g[off])) : 0.f;
        }
        for (int e = tid; e < C * DV; e += SIMT_THREADS) {
            const int t = e / DV, jl = e % DV;
            v_s[e] = t < n ? to_f32(v[(size_t)(c0 + t) * D + j0 + jl]) : 0.f;
        }
        __syncthreads();
        // 2. In-chunk inclusive cumulative sum of the log gates.
        if (tid < D) {
            float run = 0.f;
            for (int t = 0; t < C; ++t) {
                run += b_s[t * LD + tid];
                b_s[t * LD + tid] = run;
            }
        }
        __syncthreads();
        // 3. Intra-chunk decayed scores A[t][s] for s <= t (exact exponentials).
        for (int e = tid; e < C * C; e += SIMT_THREADS) {
            const int t = e / C, s = e % C;
            float acc = 0.f;
            if (s <= t && t < n) {
                for (int i = 0; i < D; ++i)
                    acc += q_s[t * LD + i] * k_s[s * LD + i] * expf(b_s[t * LD + i] - b_s[s * LD + i]);
            }
            A_s[e] = acc;
        }
        __syncthreads();
        // 4. Output rows: one warp per row.
        for (int t = warp; t < n; t += SIMT_WARPS) {
            float acc[JPL];
#pragma unroll
            for (int jj = 0; jj < JPL; ++jj) acc[jj] = 0.f;
            // inter-chunk readout (q * e^{b}) S
            for (int i = 0; i < D; ++i) {
                const float coef = q_s[t * LD + i] * expf(b_s[t * LD + i]);
#pragma unroll
                for (int jj = 0; jj < JPL; ++jj) acc[jj] += coef * S_s[i * DV + lane + 32 * jj];
            }
            // intra-chunk
            for (int s = 0; s <= t; ++s) {
                const float as = A_s[t * C + s];
#pragma unroll
                for (int jj = 0; jj < JPL; ++jj) acc[jj] += as * v_s[s * DV + lane + 32 * jj];
            }
            // anchor: window tau in [max(-nvalid, t_g - w + 1), t_g] plus m sinks
            const int tg = c0 + t;
            const int first = max(-nvalid, tg - w + 1);
            const int nk = tg - first + 1;
            for (int c = 0; c < nk + m; ++c) {
                float part = 0.f;
                if (c < nk) {
                    const int tau = first + c;
                    if (tau >= c0) {
                        for (int i = lane; i < D; i += 32) part += q_s[t * LD + i] * k_s[(tau - c0) * LD + i];
                    } else {
                        const T *kr = tau >= 0 ? k + (size_t)tau * D : history_row(ring_k, p0, tau, nvalid, w, D);
                        for (int i = lane; i < D; i += 32) part += q_s[t * LD + i] * to_f32(kr[i]);
                    }
                } else {
                    for (int i = lane; i < D; i += 32) part += q_s[t * LD + i] * to_f32(mu[(size_t)(c - nk) * D + i]);
                }
                part = warp_sum(part);
                if (lane == 0) sc[c] = part;
            }
            __syncwarp();
            float M = -INFINITY;
            for (int c = lane; c < nk + m; c += 32) M = fmaxf(M, sc[c]);
            M = warp_max(M);
            float Z = 0.f;
            for (int c = lane; c < nk + m; c += 32) Z += expf(sc[c] - M);
            Z = warp_sum(Z);
            const float scale = head_alpha(a.alpha_h, a.alpha, h) / Z;
            for (int c = 0; c < nk; ++c) {
                const int tau = first + c;
                const float pc = expf(sc[c] - M) * scale;
#pragma unroll
                for (int jj = 0; jj < JPL; ++jj) {
                    const int jl = lane + 32 * jj, j = j0 + jl;
                    const float vv = tau >= c0 ? v_s[(tau - c0) * DV + jl]
                                     : tau >= 0 ? to_f32(v[(size_t)tau * D + j])
                                                : to_f32(history_row(ring_v, p0, tau, nvalid, w, D)[j]);
                    acc[jj] += pc * vv;
                }
            }
#pragma unroll
            for (int jj = 0; jj < JPL; ++jj) y[(size_t)tg * D + j0 + lane + 32 * jj] = from_f32<T>(acc[jj]);
            __syncwarp();
        }
        __syncthreads();
        // 5. State update: k <- k * e^{b_last - b}; S <- diag(e^{b_last}) S + k^T v.
        for (int e = tid; e < C * D; e += SIMT_THREADS) {
            const int s = e / D, i = e % D;
            k_s[s * LD + i] = s < n ? k_s[s * LD + i] * expf(b_s[(n - 1) * LD + i] - b_s[s * LD + i]) : 0.f;
        }
        __syncthreads();
        {
            constexpr int JB = 16;
            for (int e = tid; e < D * (DV / JB); e += SIMT_THREADS) {
                const int i = e / (DV / JB), jb = (e % (DV / JB)) * JB;
                const float dec = expf(b_s[(n - 1) * LD + i]);
                float acc[JB];
#pragma unroll
                for (int jj = 0; jj < JB; ++jj) acc[jj] = dec * S_s[i * DV + jb + jj];
                for (int s = 0; s < n; ++s) {
                    const float kl = k_s[s * LD + i];
#pragma unroll
                    for (int jj = 0; jj < JB; ++jj) acc[jj] += kl * v_s[s * DV + jb + jj];
                }
#pragma unroll
                for (int jj = 0; jj < JB; ++jj) S_s[i * DV + jb + jj] = acc[jj];
            }
        }
    }
    __syncthreads();
    // 6. State out: S (this CTA's columns); with one CTA per unit also the
    //    last min(L, w) tokens into the ring (token p0 + tau in slot
    //    (p0 + tau) % w) and pos = L (a continued prompt advanced pos when it
    //    started).  With value slices the ring may still be read as window
    //    history by another slice of the unit, so ring_handoff_kernel writes
    //    it after this kernel.
    if (a.S_out) {
        float *So = a.S_out + (size_t)unit * D * D;
        for (int e = tid; e < D * DV; e += SIMT_THREADS) So[(e / DV) * D + j0 + e % DV] = S_s[e];
    }
    if (a.S_out && NSL == 1) {
        T *rk = static_cast<T *>(a.ring_k) + (size_t)unit * w * D;
        T *rv = static_cast<T *>(a.ring_v) + (size_t)unit * w * D;
        const int first = max(0, L - w);
        for (int e = tid; e < (L - first) * D; e += SIMT_THREADS) {
            const int tau = first + e / D, i = e % D;
            const size_t slot = (size_t)((p0 + tau) % w);
            rk[slot * D + i] = k[(size_t)tau * D + i];
            rv[slot * D + i] = v[(size_t)tau * D + i];
        }
        if (!a.cont && h == 0 && tid == 0) a.pos[unit / a.H] = L;
    }
}

// The ring and pos hand-off of a prefill that ran with value slices: one CTA
// per (batch, head) unit, after the prefill kernel.  A continued prompt
// advanced pos by L when it started, so its start position is pos - L.
template <typename T, int D>
__global__ void __launch_bounds__(SIMT_THREADS) ring_handoff_kernel(PrefillArgs a)
{
    const int unit = blockIdx.x, L = a.L, w = a.w;
    const int64_t p0 = a.cont ? a.pos[unit / a.H] - L : 0;
    const size_t kvbase = (size_t)kv_unit(unit, a.H, a.group) * L * D;
    const T *k = static_cast<const T *>(a.k) + kvbase, *v = static_cast<const T *>(a.v) + kvbase;
    T *rk = static_cast<T *>(a.ring_k) + (size_t)unit * w * D, *rv = static_cast<T *>(a.ring_v) + (size_t)unit * w * D;
    const int first = max(0, L - w);
    const int p0w = (int)(p0 % w);
    for (int e = threadIdx.x; e < (L - first) * D; e += blockDim.x) {
        const int tau = first + e / D, i = e % D;
        const size_t slot = (size_t)((p0w + tau) % w);
        rk[slot * D + i] = k[(size_t)tau * D + i];
        rv[slot * D + i] = v[(size_t)tau * D + i];
    }
    if (!a.cont && unit % a.H == 0 && threadIdx.x == 0) a.pos[unit / a.H] = L;
}

}  // namespace lizard
