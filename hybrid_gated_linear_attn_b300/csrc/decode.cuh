// decode.cuh -- one decode step of the Lizard operator (memory-bound).
//
// Lizard (gist.science/de) section 2 item 1: constant-memory inference by
// incremental updates of the hidden state; item 2: the anchor window plus
// meta-memory sinks; item 3: y = yg + alpha * ya.
//
// One CTA per (sequence, head).  The d x d fp32 state S dominates the bytes
// (64 KiB in and 64 KiB out per head at d = 128), so the kernel is laid out
// for streaming S: a warp covers one full row of S (512 B at d = 128) with
// 16-byte vector loads, each thread keeps D/RG rows x 4 columns in registers,
// and every S load is issued before the window softmax is computed so the
// HBM latency overlaps that work.  yg = q S and the anchor sum are reduced
// across row groups through one shared-memory pass.
#pragma once

#include "common.cuh"

namespace lizard {

struct DecodeArgs {
    const void *q, *k, *v, *g, *mu;
    void *y;
    float *S;
    void *ring_k, *ring_v;
    const int64_t *pos;
    float alpha;
    int B, H, w, m;
};

constexpr int DECODE_THREADS = 512;

template <int D>
__host__ __device__ constexpr int decode_row_groups() { return DECODE_THREADS / (D / 4); }

template <int D>
size_t decode_smem_bytes(int w, int m)
{
    return sizeof(float) * (4 * D + decode_row_groups<D>() * D + w + m + 8);
}

template <typename T, int D>
__global__ void __launch_bounds__(DECODE_THREADS, 2) decode_step_kernel(DecodeArgs a)
{
    constexpr int CQ = D / 4;                 // column quads per row
    constexpr int RG = DECODE_THREADS / CQ;   // row groups
    constexpr int RPT = D / RG;               // rows of S per thread
    constexpr int NW = DECODE_THREADS / 32;
    static_assert(RG * CQ == DECODE_THREADS && RPT * RG == D, "decode tiling");

    const int unit = blockIdx.x;
    const int b = unit / a.H, h = unit % a.H;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int cq = tid % CQ, rg = tid / CQ;

    extern __shared__ float sm[];
    float *q_s = sm, *k_s = q_s + D, *v_s = k_s + D, *gam_s = v_s + D;
    float *red = gam_s + D;          // [RG][D]
    float *sc = red + RG * D;        // [w + m] logits, then weights
    float *stat = sc + a.w + a.m;    // M, 1/Z

    const int64_t p = a.pos[b];
    const int w = a.w, m = a.m;
    if (p < 0) {  // not a state this library wrote: record it, touch nothing
        if (tid == 0) atomicExch(&g_device_error, DEV_BAD_POS);
        return;
    }

    // 1. Issue the state loads first (the bulk of the bytes).
    float4 *Sg = reinterpret_cast<float4 *>(a.S + (size_t)unit * D * D);
    float4 s_reg[RPT];
#pragma unroll
    for (int r = 0; r < RPT; ++r) s_reg[r] = Sg[(size_t)(rg + r * RG) * CQ + cq];

    // 2. Current token into shared memory; gate gamma = sigmoid(g).
    const T *q = static_cast<const T *>(a.q) + (size_t)unit * D;
    const T *k = static_cast<const T *>(a.k) + (size_t)unit * D;
    const T *v = static_cast<const T *>(a.v) + (size_t)unit * D;
    const T *g = static_cast<const T *>(a.g) + (size_t)unit * D;
    if (tid < D) {
        q_s[tid] = to_f32(q[tid]);
        k_s[tid] = to_f32(k[tid]);
        v_s[tid] = to_f32(v[tid]);
        gam_s[tid] = expf(log_sigmoid(to_f32(g[tid])));
    }
    __syncthreads();

    // 3. Window logits: history tokens first .. p-1 from the ring, then the
    //    current token, then the m meta keys.  One warp per logit.
    const int64_t first = p - w + 1 > 0 ? p - w + 1 : 0;
    const int n = (int)(p - first) + 1;
    const T *ring_k = static_cast<const T *>(a.ring_k) + (size_t)unit * w * D;
    const T *ring_v = static_cast<const T *>(a.ring_v) + (size_t)unit * w * D;
    const T *mu = static_cast<const T *>(a.mu) + (size_t)h * m * D;
    for (int c = warp; c < n + m; c += NW) {
        float part = 0.f;
        if (c < n - 1) {
            const T *kr = ring_k + (size_t)((first + c) % w) * D;
            for (int i = lane; i < D; i += 32) part += q_s[i] * to_f32(kr[i]);
        } else if (c == n - 1) {
            for (int i = lane; i < D; i += 32) part += q_s[i] * k_s[i];
        } else {
            const T *mr = mu + (size_t)(c - n) * D;
            for (int i = lane; i < D; i += 32) part += q_s[i] * to_f32(mr[i]);
        }
        part = warp_sum(part);
        if (lane == 0) sc[c] = part;
    }
    __syncthreads();
    if (warp == 0) {
        float M = -INFINITY;
        for (int c = lane; c < n + m; c += 32) M = fmaxf(M, sc[c]);
        M = warp_max(M);
        float Z = 0.f;
        for (int c = lane; c < n + m; c += 32) Z += expf(sc[c] - M);
        Z = warp_sum(Z);
        if (lane == 0) { stat[0] = M; stat[1] = 1.f / Z; }
    }
    __syncthreads();
    const float M = stat[0], scale = a.alpha * stat[1];

    // 4. Anchor partial: this row group's share of the window keys.
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int c = rg; c < n; c += RG) {
        const float pc = expf(sc[c] - M) * scale;
        float4 vv = c < n - 1 ? load4(ring_v + (size_t)((first + c) % w) * D + cq * 4)
                              : make_float4(v_s[cq * 4], v_s[cq * 4 + 1], v_s[cq * 4 + 2], v_s[cq * 4 + 3]);
        acc.x += pc * vv.x; acc.y += pc * vv.y; acc.z += pc * vv.z; acc.w += pc * vv.w;
    }

    // 5. State update S <- diag(gamma) S + k^T v and readout yg = q S.
    const float4 vq = make_float4(v_s[cq * 4], v_s[cq * 4 + 1], v_s[cq * 4 + 2], v_s[cq * 4 + 3]);
#pragma unroll
    for (int r = 0; r < RPT; ++r) {
        const int row = rg + r * RG;
        const float gi = gam_s[row], ki = k_s[row], qi = q_s[row];
        float4 s = s_reg[r];
        s.x = gi * s.x + ki * vq.x;
        s.y = gi * s.y + ki * vq.y;
        s.z = gi * s.z + ki * vq.z;
        s.w = gi * s.w + ki * vq.w;
        Sg[(size_t)row * CQ + cq] = s;
        acc.x += qi * s.x; acc.y += qi * s.y; acc.z += qi * s.z; acc.w += qi * s.w;
    }
    *reinterpret_cast<float4 *>(red + rg * D + cq * 4) = acc;

    // 6. Ring slot p % w takes the current token (it held token p - w, which
    //    is outside this step's window, so no reader above touched it).
    if (tid < D) {
        T *rk = static_cast<T *>(a.ring_k) + ((size_t)unit * w + (size_t)(p % w)) * D;
        T *rv = static_cast<T *>(a.ring_v) + ((size_t)unit * w + (size_t)(p % w)) * D;
        rk[tid] = k[tid];
        rv[tid] = v[tid];
    }
    __syncthreads();
    if (tid < D) {
        float y = 0.f;
#pragma unroll 8
        for (int r = 0; r < RG; ++r) y += red[r * D + tid];
        static_cast<T *>(a.y)[(size_t)unit * D + tid] = from_f32<T>(y);
    }
}

__global__ void advance_pos_kernel(int64_t *pos, int B)
{
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < B) pos[i] += 1;
}

}  // namespace lizard
