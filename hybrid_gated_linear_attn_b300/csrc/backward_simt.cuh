// backward_simt.cuh -- gradients of the Lizard operator (dq, dk, dv, dg,
// d mu, d alpha) on CUDA cores, exact fp32, for prompts that start from the
// empty state (training).
//
// Forward (Lizard, gist.science/de section 2 items 1-3):
//   S_t = diag(gamma_t) S_{t-1} + k_t^T v_t,  gamma = sigmoid(g),  yg_t = q_t S_t
//   ya_t = sum_s p_ts v_s,  p over the window keys s and the meta keys mu_j
//          (value 0) of softmax(q_t k_s, q_t mu_j)
//   y_t  = yg_t + alpha ya_t
// With B_t[i] = sum_{r<=t} log gamma_r[i] and dy = dLoss/dy:
//   dq_t  = sum_{s<=t} (dy_t . v_s) k_s e^{B_t - B_s}            (gate)
//         + sum_s da_ts k_s + sum_j dc_tj mu_j                   (anchor)
//   dk_s  = sum_{t>=s} (dy_t . v_s) q_t e^{B_t - B_s} + sum_t da_ts q_t
//   dv_s  = sum_{t>=s} (sum_i q_t k_s e^{B_t - B_s}) dy_t + alpha sum_t p_ts dy_t
//   da_ts = p_ts (alpha dy_t . v_s - D_t),  dc_tj = p_tj (0 - D_t),
//   D_t   = alpha dy_t . ya_t,  d mu_j = sum_t dc_tj q_t,  d alpha = sum_t dy_t . ya_t
//   dlog gamma_t = sum_{r>=t} (q_r * dq_r - k_r * dk_r)  (gate parts only; each
//          term of yg depends on B through B_t - B_s), dg = dlog gamma * sigmoid(-g).
// The chunked evaluation (C = 32 tokens, b = in-chunk prefix of log gamma,
// the log-space form of the page's "Hardware-bewusster Algorithmus") keeps
// every exponent <= 0:
//   forward sweep, S = state before the chunk:
//     dq_t = e^{b_t} (S dy_t) + sum_{s<=t in chunk} (dy_t . v_s) k_s e^{b_t - b_s}
//     S   <- diag(e^{b_last}) S + sum_s (k_s e^{b_last - b_s})^T v_s
//   reverse sweep, H = dLoss/d(state after the chunk):
//     dk_s = e^{b_last - b_s} (H v_s) + sum_{t>=s in chunk} (dy_t . v_s) q_t e^{b_t - b_s}
//     dv_s = (k_s e^{b_last - b_s}) H + sum_{t>=s in chunk} A_ts dy_t
//     H   <- diag(e^{b_last}) H + sum_t (q_t e^{b_t})^T dy_t
// The anchor part of dq is done per query row in the forward sweep, which
// also stores each row's log-normaliser and D_t; the anchor parts of dk and
// dv are gathered per key in the reverse sweep from those.
// One CTA per (batch, head) unit; scratch per unit: q * dq_gate [L][D] and
// the two row statistics [L] (fp32), d mu partial [m][D], d alpha partial.
#pragma once

#include "common.cuh"

namespace lizard {

struct BackwardArgs {
    const void *q, *k, *v, *g, *mu, *dy;
    void *dq, *dk, *dv, *dg;
    float alpha;
    int B, H, L, w, m;
    float *xq;          // [units][L][D]  q * dq (gate branch)
    float *lse, *drow;  // [units][L]     log-normaliser and D_t of each row
    float *dmu_part;    // [units][m][D]
    float *dalpha_part; // [units]
    const float *alpha_h;  // per-head anchor weights (null: alpha)
    int group;             // query heads per key/value head (k, v hold B x H / group heads)
};

constexpr int BW_C = 32;  // chunk length
constexpr int BW_THREADS = 256;
constexpr int BW_WARPS = BW_THREADS / 32;

template <int D>
size_t backward_simt_smem_bytes(int w, int m)
{
    const size_t LD = D + 1, LC = BW_C + 1;
    return sizeof(float) * ((size_t)D * LD + 6 * (size_t)BW_C * LD + 2 * (size_t)BW_C * LC + 2 * (size_t)BW_C * D +
                            (size_t)BW_WARPS * 2 * (w + m) + (size_t)m * D + D + BW_WARPS);
}

template <typename T, int D>
__global__ void __launch_bounds__(BW_THREADS, 1) backward_simt_kernel(BackwardArgs a)
{
    constexpr int C = BW_C, LD = D + 1, LC = C + 1;
    constexpr int TG = BW_THREADS / D;  // token groups (threads per feature index)
    constexpr int TPG = C / TG;         // tokens per group
    constexpr int JPL = D / 32;         // features per lane
    constexpr int JB = 16;              // state columns per thread in the state updates
    const int unit = blockIdx.x, h = unit % a.H;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int L = a.L, w = a.w, m = a.m;
    const float alpha = head_alpha(a.alpha_h, a.alpha, h);

    extern __shared__ float sm[];
    float *S = sm;                    // [D][LD] state (forward sweep) / state gradient (reverse sweep)
    float *q_s = S + D * LD;          // [C][LD]
    float *k_s = q_s + C * LD;
    float *b_s = k_s + C * LD;        // in-chunk prefix of log gamma
    float *v_s = b_s + C * LD;
    float *dy_s = v_s + C * LD;
    float *kl_s = dy_s + C * LD;      // k e^{b_last - b}
    float *A_s = kl_s + C * LD;       // [C][LC] intra-chunk decayed scores
    float *dA_s = A_s + C * LC;       // [C][LC] dy_t . v_s
    float *o1 = dA_s + C * LC;        // [C][D] dq (forward) / dk (reverse)
    float *o2 = o1 + C * D;           // [C][D] dv (reverse)
    float *sc_all = o2 + C * D;       // [warps][2 (w + m)] scores, then dp
    float *dmu_s = sc_all + BW_WARPS * 2 * (w + m);  // [m][D]
    float *carry = dmu_s + m * D;     // [D] sum of later tokens' dlog gamma terms
    float *dal_s = carry + D;         // [warps]
    float *sc = sc_all + warp * 2 * (w + m), *dp = sc + (w + m);

    const size_t base = (size_t)unit * L * D;
    const T *q = static_cast<const T *>(a.q) + base;
    const size_t kvbase = (size_t)kv_unit(unit, a.H, a.group) * L * D;
    const T *k = static_cast<const T *>(a.k) + kvbase;
    const T *v = static_cast<const T *>(a.v) + kvbase;
    const T *g = static_cast<const T *>(a.g) + base;
    const T *dy = static_cast<const T *>(a.dy) + base;
    const T *mu = static_cast<const T *>(a.mu) + (size_t)h * m * D;
    T *dq = static_cast<T *>(a.dq) + base;
    T *dk = static_cast<T *>(a.dk) + base;
    T *dv = static_cast<T *>(a.dv) + base;
    T *dg = static_cast<T *>(a.dg) + base;
    float *xq = a.xq + base;
    float *lse = a.lse + (size_t)unit * L, *drow = a.drow + (size_t)unit * L;

    for (int e = tid; e < D * LD; e += BW_THREADS) S[e] = 0.f;
    for (int e = tid; e < m * D; e += BW_THREADS) dmu_s[e] = 0.f;
    for (int e = tid; e < D; e += BW_THREADS) carry[e] = 0.f;
    float dal = 0.f;  // this warp's part of d alpha (lane 0)

    // Chunk tiles in fp32 (rows >= n zero: no token, no decay) and the
    // in-chunk prefix sums of log gamma.
    auto load_chunk = [&](int c0, int n) {
        for (int e = tid; e < C * D; e += BW_THREADS) {
            const int t = e / D, i = e % D;
            const bool ok = t < n;
            const size_t off = (size_t)(c0 + t) * D + i;
            q_s[t * LD + i] = ok ? to_f32(q[off]) : 0.f;
            k_s[t * LD + i] = ok ? to_f32(k[off]) : 0.f;
            v_s[t * LD + i] = ok ? to_f32(v[off]) : 0.f;
            dy_s[t * LD + i] = ok ? to_f32(dy[off]) : 0.f;
            b_s[t * LD + i] = ok ? log_sigmoid(to_f32(g[off])) : 0.f;
        }
        __syncthreads();
        if (tid < D) {
            float run = 0.f;
            for (int t = 0; t < C; ++t) {
                run += b_s[t * LD + tid];
                b_s[t * LD + tid] = run;
            }
        }
        __syncthreads();
    };
    // kl = k e^{b_last - b} (rows >= n zero).
    auto fill_kl = [&](int n) {
        for (int e = tid; e < C * D; e += BW_THREADS) {
            const int s = e / D, i = e % D;
            kl_s[s * LD + i] = s < n ? k_s[s * LD + i] * expf(b_s[(n - 1) * LD + i] - b_s[s * LD + i]) : 0.f;
        }
    };
    // X <- diag(e^{b_last}) X + sum_{s<n} lhs_s^T rhs_s, X = S (or H).  lhs
    // row s scaled by e^{b_s} when `scale_b` (the q e^{b} of the reverse sweep).
    auto update_state = [&](int n, const float *lhs, const float *rhs, bool scale_b) {
        for (int e = tid; e < D * (D / JB); e += BW_THREADS) {
            const int i = e % D, j0 = (e / D) * JB;
            const float dec = expf(b_s[(n - 1) * LD + i]);
            float acc[JB];
#pragma unroll
            for (int jj = 0; jj < JB; ++jj) acc[jj] = dec * S[i * LD + j0 + jj];
            for (int s = 0; s < n; ++s) {
                const float l = scale_b ? lhs[s * LD + i] * expf(b_s[s * LD + i]) : lhs[s * LD + i];
#pragma unroll
                for (int jj = 0; jj < JB; ++jj) acc[jj] += l * rhs[s * LD + j0 + jj];
            }
#pragma unroll
            for (int jj = 0; jj < JB; ++jj) S[i * LD + j0 + jj] = acc[jj];
        }
    };

    // ------------------------------------------------------------ forward sweep
    for (int c0 = 0; c0 < L; c0 += C) {
        const int n = min(C, L - c0);
        __syncthreads();
        load_chunk(c0, n);
        // dA[t][s] = dy_t . v_s for s <= t
        for (int e = tid; e < C * C; e += BW_THREADS) {
            const int t = e / C, s = e % C;
            float acc = 0.f;
            if (s <= t && t < n)
                for (int j = 0; j < D; ++j) acc += dy_s[t * LD + j] * v_s[s * LD + j];
            dA_s[t * LC + s] = acc;
        }
        __syncthreads();
        // gate part of dq (inter-chunk term from S, then intra-chunk), and q * dq
        {
            const int i = tid % D, tg = tid / D;
            float acc[TPG];
#pragma unroll
            for (int tt = 0; tt < TPG; ++tt) acc[tt] = 0.f;
            for (int j = 0; j < D; ++j) {
                const float sij = S[i * LD + j];
#pragma unroll
                for (int tt = 0; tt < TPG; ++tt) acc[tt] += sij * dy_s[(tg * TPG + tt) * LD + j];
            }
#pragma unroll
            for (int tt = 0; tt < TPG; ++tt) {
                const int t = tg * TPG + tt;
                const float bt = b_s[t * LD + i];
                float r = acc[tt] * expf(bt);
                for (int s = 0; s <= t; ++s) r += dA_s[t * LC + s] * k_s[s * LD + i] * expf(bt - b_s[s * LD + i]);
                if (t >= n) r = 0.f;
                o1[t * D + i] = r;
                if (t < n) xq[(size_t)(c0 + t) * D + i] = q_s[t * LD + i] * r;
            }
        }
        __syncthreads();
        // anchor: one warp per query row
        for (int t = warp; t < n; t += BW_WARPS) {
            const int tg = c0 + t;
            const int first = max(0, tg - w + 1);
            const int nk = tg - first + 1;
            for (int c = 0; c < nk + m; ++c) {
                float ps = 0.f, pd = 0.f;
                if (c < nk) {
                    const int tau = first + c;
                    if (tau >= c0) {
                        for (int i = lane; i < D; i += 32) {
                            ps += q_s[t * LD + i] * k_s[(tau - c0) * LD + i];
                            pd += dy_s[t * LD + i] * v_s[(tau - c0) * LD + i];
                        }
                    } else {
                        for (int i = lane; i < D; i += 32) {
                            ps += q_s[t * LD + i] * to_f32(k[(size_t)tau * D + i]);
                            pd += dy_s[t * LD + i] * to_f32(v[(size_t)tau * D + i]);
                        }
                    }
                } else {
                    for (int i = lane; i < D; i += 32) ps += q_s[t * LD + i] * to_f32(mu[(size_t)(c - nk) * D + i]);
                }
                ps = warp_sum(ps);
                pd = warp_sum(pd);
                if (lane == 0) {
                    sc[c] = ps;
                    dp[c] = pd;  // dy_t . v_s
                }
            }
            __syncwarp();
            float M = -INFINITY;
            for (int c = lane; c < nk + m; c += 32) M = fmaxf(M, sc[c]);
            M = warp_max(M);
            float Z = 0.f, pdp = 0.f;
            for (int c = lane; c < nk + m; c += 32) {
                const float p = expf(sc[c] - M);
                Z += p;
                if (c < nk) pdp += p * dp[c];
            }
            Z = warp_sum(Z);
            pdp = warp_sum(pdp);
            const float invZ = 1.f / Z;
            const float dyya = pdp * invZ;  // dy_t . ya_t
            const float Dt = alpha * dyya;
            if (lane == 0) {
                dal += dyya;
                lse[tg] = M + logf(Z);
                drow[tg] = Dt;
            }
            float acc[JPL];
#pragma unroll
            for (int jj = 0; jj < JPL; ++jj) acc[jj] = 0.f;
            for (int c = 0; c < nk + m; ++c) {
                const float p = expf(sc[c] - M) * invZ;
                const float ds = p * ((c < nk ? alpha * dp[c] : 0.f) - Dt);
                if (c < nk) {
                    const int tau = first + c;
#pragma unroll
                    for (int jj = 0; jj < JPL; ++jj) {
                        const int i = lane + 32 * jj;
                        acc[jj] += ds * (tau >= c0 ? k_s[(tau - c0) * LD + i] : to_f32(k[(size_t)tau * D + i]));
                    }
                } else {
                    const int j = c - nk;
#pragma unroll
                    for (int jj = 0; jj < JPL; ++jj) {
                        const int i = lane + 32 * jj;
                        acc[jj] += ds * to_f32(mu[(size_t)j * D + i]);
                        atomicAdd(&dmu_s[j * D + i], ds * q_s[t * LD + i]);
                    }
                }
            }
#pragma unroll
            for (int jj = 0; jj < JPL; ++jj) o1[t * D + lane + 32 * jj] += acc[jj];
            __syncwarp();
        }
        __syncthreads();
        for (int e = tid; e < n * D; e += BW_THREADS) dq[(size_t)c0 * D + e] = from_f32<T>(o1[e]);
        fill_kl(n);
        __syncthreads();
        update_state(n, kl_s, v_s, false);
    }
    __syncthreads();
    for (int e = tid; e < m * D; e += BW_THREADS) a.dmu_part[(size_t)unit * m * D + e] = dmu_s[e];
    if (lane == 0) dal_s[warp] = dal;
    // ------------------------------------------------------------ reverse sweep
    for (int e = tid; e < D * LD; e += BW_THREADS) S[e] = 0.f;  // now H = dLoss/dS
    __syncthreads();
    if (tid == 0) {
        float s = 0.f;
        for (int i = 0; i < BW_WARPS; ++i) s += dal_s[i];
        a.dalpha_part[unit] = s;
    }
    const int nchunks = (L + C - 1) / C;
    for (int ci = nchunks - 1; ci >= 0; --ci) {
        const int c0 = ci * C, n = min(C, L - c0);
        __syncthreads();
        load_chunk(c0, n);
        // A[t][s] = sum_i q_t k_s e^{b_t - b_s} and dA[t][s] = dy_t . v_s, s <= t
        for (int e = tid; e < C * C; e += BW_THREADS) {
            const int t = e / C, s = e % C;
            float acc = 0.f, dacc = 0.f;
            if (s <= t && t < n) {
                for (int i = 0; i < D; ++i) {
                    acc += q_s[t * LD + i] * k_s[s * LD + i] * expf(b_s[t * LD + i] - b_s[s * LD + i]);
                    dacc += dy_s[t * LD + i] * v_s[s * LD + i];
                }
            }
            A_s[t * LC + s] = acc;
            dA_s[t * LC + s] = dacc;
        }
        fill_kl(n);
        __syncthreads();
        // gate parts of dk (o1) and dv (o2)
        {
            const int i = tid % D, sg = tid / D;
            float acc[TPG], acc2[TPG];
#pragma unroll
            for (int ss = 0; ss < TPG; ++ss) acc[ss] = acc2[ss] = 0.f;
            for (int j = 0; j < D; ++j) {
                const float hij = S[i * LD + j];  // H[i][j]
                const float hji = S[j * LD + i];  // H[j][i]: feature i is a value column here
#pragma unroll
                for (int ss = 0; ss < TPG; ++ss) {
                    acc[ss] += hij * v_s[(sg * TPG + ss) * LD + j];
                    acc2[ss] += kl_s[(sg * TPG + ss) * LD + j] * hji;
                }
            }
            const float bl = b_s[(n - 1) * LD + i];
#pragma unroll
            for (int ss = 0; ss < TPG; ++ss) {
                const int s = sg * TPG + ss;
                const float bsi = b_s[s * LD + i];
                float r = acc[ss] * expf(bl - bsi), r2 = acc2[ss];
                for (int t = s; t < n; ++t) {
                    r += dA_s[t * LC + s] * q_s[t * LD + i] * expf(b_s[t * LD + i] - bsi);
                    r2 += A_s[t * LC + s] * dy_s[t * LD + i];
                }
                o1[s * D + i] = s < n ? r : 0.f;
                o2[s * D + i] = s < n ? r2 : 0.f;
            }
        }
        __syncthreads();
        // dlog gamma = reverse prefix of (q dq - k dk) over all later tokens; dg
        if (tid < D) {
            const int i = tid;
            float run = carry[i];
            for (int t = n - 1; t >= 0; --t) {
                run += xq[(size_t)(c0 + t) * D + i] - k_s[t * LD + i] * o1[t * D + i];
                const float sgn = expf(log_sigmoid(-to_f32(g[(size_t)(c0 + t) * D + i])));  // sigmoid(-g)
                dg[(size_t)(c0 + t) * D + i] = from_f32<T>(run * sgn);
            }
            carry[i] = run;
        }
        __syncthreads();
        // anchor parts of dk, dv: one warp per key, over the queries whose
        // window holds it (t = s .. s + w - 1)
        for (int s = warp; s < n; s += BW_WARPS) {
            const int sg = c0 + s;
            const int tend = min(L, sg + w);
            float ak[JPL], av[JPL];
#pragma unroll
            for (int jj = 0; jj < JPL; ++jj) ak[jj] = av[jj] = 0.f;
            for (int t = sg; t < tend; ++t) {
                const bool here = t - c0 < n;
                float ps = 0.f, pd = 0.f;
                float qv[JPL], dyv[JPL];
#pragma unroll
                for (int jj = 0; jj < JPL; ++jj) {
                    const int i = lane + 32 * jj;
                    qv[jj] = here ? q_s[(t - c0) * LD + i] : to_f32(q[(size_t)t * D + i]);
                    dyv[jj] = here ? dy_s[(t - c0) * LD + i] : to_f32(dy[(size_t)t * D + i]);
                    ps += qv[jj] * k_s[s * LD + i];
                    pd += dyv[jj] * v_s[s * LD + i];
                }
                ps = warp_sum(ps);
                pd = warp_sum(pd);
                const float p = expf(ps - lse[t]);
                const float ds = p * (alpha * pd - drow[t]);
#pragma unroll
                for (int jj = 0; jj < JPL; ++jj) {
                    ak[jj] += ds * qv[jj];
                    av[jj] += alpha * p * dyv[jj];
                }
            }
#pragma unroll
            for (int jj = 0; jj < JPL; ++jj) {
                o1[s * D + lane + 32 * jj] += ak[jj];
                o2[s * D + lane + 32 * jj] += av[jj];
            }
        }
        __syncthreads();
        for (int e = tid; e < n * D; e += BW_THREADS) {
            dk[(size_t)c0 * D + e] = from_f32<T>(o1[e]);
            dv[(size_t)c0 * D + e] = from_f32<T>(o2[e]);
        }
        update_state(n, q_s, dy_s, true);
    }
}

// d mu[h] = sum over the batch of the units' partials; d alpha = sum over all
// units (per_head: d alpha[h] = sum over the batch, by block 0's first H
// threads).  grid.x covers H * m * D elements; block 0 also sums d alpha.
__global__ void backward_reduce_kernel(const float *dmu_part, const float *dalpha_part, int B, int H, int mD,
                                       float *dmu, float *dalpha, int per_head)
{
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    if (dmu && e < H * mD) {
        const int h = e / mD, r = e % mD;
        float s = 0.f;
        for (int b = 0; b < B; ++b) s += dmu_part[((size_t)b * H + h) * mD + r];
        dmu[e] = s;
    }
    if (blockIdx.x == 0 && per_head) {
        for (int hh = threadIdx.x; hh < H; hh += blockDim.x) {
            float s = 0.f;
            for (int b = 0; b < B; ++b) s += dalpha_part[(size_t)b * H + hh];
            dalpha[hh] = s;
        }
    } else if (blockIdx.x == 0) {
        __shared__ float red[256];
        float s = 0.f;
        for (long long u = threadIdx.x; u < (long long)B * H; u += blockDim.x) s += dalpha_part[u];
        red[threadIdx.x] = s;
        __syncthreads();
        for (int o = blockDim.x / 2; o > 0; o >>= 1) {
            if ((int)threadIdx.x < o) red[threadIdx.x] += red[threadIdx.x + o];
            __syncthreads();
        }
        if (threadIdx.x == 0) *dalpha = red[0];
    }
}

// Grouped key/value heads: dk, dv of key/value head hk are the sums over
// the group's query heads (the key and value feed every head of the group):
// dst[b][hk][e] = sum_j src[b][hk group + j][e], in fp32, rounded once.
// grid-stride over B * Hkv * LD elements (LD = L * D).
template <typename T>
__global__ void gqa_reduce_kernel(const T *src, T *dst, int B, int H, int group, long long LD)
{
    const int Hkv = H / group;
    const long long n = (long long)B * Hkv * LD;
    for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < n; e += (long long)gridDim.x * blockDim.x) {
        const long long r = e % LD, bh = e / LD;
        const long long b = bh / Hkv, hk = bh % Hkv;
        float s = 0.f;
        for (int j = 0; j < group; ++j) s += to_f32(src[((b * H) + hk * group + j) * LD + r]);
        dst[e] = from_f32<T>(s);
    }
}

}  // namespace lizard
