// decode.cuh -- one decode step of the Lizard operator (memory-bound).
//
// Lizard (gist.science/de) section 2 item 1: constant-memory inference by
// incremental updates of the hidden state; item 2: the anchor window plus
// meta-memory sinks; item 3: y = yg + alpha * ya.
//
// Bytes per (sequence, head) at d = 128, w = 64, bf16: the fp32 state S is
// read and written (2 x 64 KiB) and the window ring's keys and values are
// read (2 x 16 KiB); everything else is a few hundred bytes.  Throughput is
// set by how many of those bytes are in flight per SM, so:
//   - each (sequence, head) unit is split over two CTAs by value columns
//     (j < d/2 and j >= d/2).  The columns of y, of the anchor sum and of
//     S are independent; the window logits need every key dimension, so
//     both CTAs compute them (the second read of the ring hits L2);
//   - small CTAs (256 threads, ~41 KiB of shared memory), four per SM;
//   - every load of a CTA is issued at its start: its half of S streams
//     into registers (coalesced 16-byte loads), and one thread moves the
//     ring keys and values, the token's q, k, v, g and the head's meta keys
//     into shared memory with bulk asynchronous copies (cp.async.bulk,
//     completion on two mbarriers -- the token and meta keys, the ring --
//     bounded waits);
//   - the state update S <- diag(gamma) S + k^T v and the readout q S come
//     first, as soon as the token is in: S goes back with 16-byte stores
//     while the ring copies land and the window is scored (7% faster than
//     scoring the window first).
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
    const float *alpha_h;  // per-head anchor weights (null: alpha)
    int group;             // query heads per key/value head (k, v are [B][H / group][D])
    // Failure-detection testing: polls of the first wait before it gives up
    // (negative: the normal limit).  The drain after a timeout always keeps
    // the normal limit, so the CTA retires only once its copies have landed.
    int first_wait_polls;
};

constexpr int DECODE_THREADS = 256;
// CTAs per unit (value-column slices): two at d <= 128, eight at d = 256, so
// that a CTA's slice of S stays 32 registers a thread.
template <int D>
__host__ __device__ constexpr int decode_split()
{
    return D > 128 ? 8 : 2;
}
constexpr int DECODE_KEY_THREADS = 8;  // threads per window key in the logit pass
constexpr uint32_t DECODE_WAIT_LIMIT = 1u << 22;
constexpr unsigned long long DECODE_POS_TICK = 1ull << 40;  // per-CTA arrival count in pos's high bits
constexpr size_t DECODE_SMEM_MAX = 232448 - 512;  // opt-in limit per block, with slack

// Shared-memory plan of the decode kernel for one (D, element size, w, m).
struct DecodePlan {
    size_t ring_bytes, tok_bytes, mu_bytes, copy_bytes, total;
    uint32_t mu_copy;
};

template <int D>
__host__ __device__ inline DecodePlan decode_plan(int esize, int w, int m)
{
    constexpr int RG = DECODE_THREADS / (D / decode_split<D>() / 4);
    DecodePlan p;
    p.ring_bytes = (size_t)w * D * esize;
    p.tok_bytes = (size_t)D * esize;                  // one of q, k, v, g
    p.mu_copy = (uint32_t)((size_t)m * D * esize);
    p.mu_bytes = ((size_t)p.mu_copy + 15) / 16 * 16;
    // ring keys | ring values | q | k | v | g | meta keys of the unit's head
    p.copy_bytes = 2 * p.ring_bytes + 4 * p.tok_bytes + p.mu_bytes;
    // then: q, k, v, gamma as fp32 [D]; logits [w + m] (rounded to 4);
    // row-group partials [RG][D / split]; stats [4]; two mbarriers (the
    // token and meta-key copies, the ring copies).
    p.total = p.copy_bytes + 4 * ((size_t)4 * D + ((w + m + 3) / 4) * 4 + (size_t)RG * (D / decode_split<D>()) + 4) + 16;
    return p;
}

__device__ __forceinline__ uint32_t dec_smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void dec_bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            dec_smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(dec_smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ bool dec_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(dec_smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Eight consecutive elements as fp32 (16-byte aligned source).
__device__ __forceinline__ void load8(const float *p, float (&x)[8])
{
    const float4 a = reinterpret_cast<const float4 *>(p)[0], b = reinterpret_cast<const float4 *>(p)[1];
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}
__device__ __forceinline__ void load8(const __nv_bfloat16 *p, float (&x)[8])
{
    const uint4 u = *reinterpret_cast<const uint4 *>(p);
    const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w4[i]));
        x[2 * i] = f.x;
        x[2 * i + 1] = f.y;
    }
}

// grid = split * B * H; CTA (unit, slice) owns value columns
// [slice * D/split, (slice + 1) * D/split).
template <typename T, int D>
__global__ void __launch_bounds__(DECODE_THREADS, 4) decode_step_kernel(DecodeArgs a)
{
    constexpr int SPLIT = decode_split<D>();
    constexpr int DH = D / SPLIT;                    // value columns of this CTA
    constexpr int CQ = DH / 4;                       // column quads per row of S
    constexpr int RG = DECODE_THREADS / CQ;          // row groups
    constexpr int RPT = D / RG;                      // rows of S per thread
    constexpr int KT = DECODE_KEY_THREADS;           // threads per key (logits)
    constexpr int DPT = D / KT;                      // dims per thread (logits)
    constexpr int KPP = DECODE_THREADS / KT;         // keys per pass (logits)
    static_assert(RG * CQ == DECODE_THREADS && RPT * RG == D && DPT % 8 == 0, "decode tiling");

    const int w = a.w, m = a.m, H = a.H;
    const int u = blockIdx.x / SPLIT, half = blockIdx.x % SPLIT, j0 = half * DH;
    const int b = u / H;
    const DecodePlan plan = decode_plan<D>((int)sizeof(T), w, m);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int cq = tid % CQ, rg = tid / CQ;

    extern __shared__ __align__(128) uint8_t dsm[];
    const T *rk = reinterpret_cast<const T *>(dsm);
    const T *rv = reinterpret_cast<const T *>(dsm + plan.ring_bytes);
    const T *tok = reinterpret_cast<const T *>(dsm + 2 * plan.ring_bytes);  // q | k | v | g
    const T *mu = reinterpret_cast<const T *>(dsm + 2 * plan.ring_bytes + 4 * plan.tok_bytes);
    float *q_s = reinterpret_cast<float *>(dsm + plan.copy_bytes);
    float *k_s = q_s + D, *v_s = k_s + D, *gam_s = v_s + D;
    float *sc = gam_s + D;                      // [w + m] logits
    float *red = sc + ((w + m + 3) / 4) * 4;    // [RG][DH]
    float *stat = red + RG * DH;                // [1]: alpha / Z
    uint64_t *bar = reinterpret_cast<uint64_t *>(stat + 4);

    // The next decode step may begin launching now; this one waits until the
    // previous kernel on the stream has finished and its writes are visible.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");

    // 1. Every load up front: the bulk copies (thread 0), this CTA's half of
    //    S into registers (all threads), the position.
    uint64_t *bar_ring = bar + 1;
    if (tid == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(dec_smem_u32(bar)) : "memory");
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(dec_smem_u32(bar_ring)) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(dec_smem_u32(bar)),
                     "r"((uint32_t)(4 * plan.tok_bytes + plan.mu_copy))
                     : "memory");
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(dec_smem_u32(bar_ring)),
                     "r"((uint32_t)(2 * plan.ring_bytes))
                     : "memory");
        const void *src[4] = {a.q, a.k, a.v, a.g};
        const size_t kvu = (size_t)kv_unit(u, H, a.group);
#pragma unroll
        for (int j = 0; j < 4; ++j)
            dec_bulk_g2s(dsm + 2 * plan.ring_bytes + j * plan.tok_bytes,
                         static_cast<const T *>(src[j]) + (j == 1 || j == 2 ? kvu : (size_t)u) * D,
                         (uint32_t)plan.tok_bytes, bar);
        if (plan.mu_copy)
            dec_bulk_g2s(dsm + 2 * plan.ring_bytes + 4 * plan.tok_bytes,
                         static_cast<const T *>(a.mu) + (size_t)(u % H) * m * D, plan.mu_copy, bar);
        dec_bulk_g2s(dsm, static_cast<const T *>(a.ring_k) + (size_t)u * w * D, (uint32_t)plan.ring_bytes, bar_ring);
        dec_bulk_g2s(dsm + plan.ring_bytes, static_cast<const T *>(a.ring_v) + (size_t)u * w * D,
                     (uint32_t)plan.ring_bytes, bar_ring);
    }
    float4 *Sg = reinterpret_cast<float4 *>(a.S + (size_t)u * D * D + j0);
    float4 s_reg[RPT];
#pragma unroll
    for (int r = 0; r < RPT; ++r) s_reg[r] = Sg[(size_t)(rg + r * RG) * (D / 4) + cq];
    // The position, read and advanced in one pass without a second kernel:
    // each of the split x H CTAs of sequence b adds 2^40 to pos[b] and takes the
    // token count from the low 40 bits of the value it got back; the CTA
    // whose addition was the last (split x H - 1 earlier ones) writes p + 1.  So
    // every CTA sees the same p whatever the scheduling order, and pos[b]
    // is p + 1 once the kernel is done.
    __shared__ long long p_sh;
    if (tid == 0) {
        const unsigned long long old =
            atomicAdd(reinterpret_cast<unsigned long long *>(const_cast<int64_t *>(a.pos) + b), DECODE_POS_TICK);
        const long long cnt = (long long)old >> 40, pv = (long long)(old & (DECODE_POS_TICK - 1));
        const int ctas = SPLIT * H;
        if (cnt < 0 || cnt >= ctas) {
            p_sh = -1;  // pos[b] was outside [0, 2^40) before the call
        } else {
            p_sh = pv;
            if (cnt == ctas - 1) atomicExch(reinterpret_cast<unsigned long long *>(const_cast<int64_t *>(a.pos) + b),
                                            (unsigned long long)(pv + 1));
        }
    }
    __syncthreads();  // p_sh, and the mbarrier's initialisation, are visible
    const int64_t p = p_sh;

    // 2. Wait for the token and meta-key copies (bounded; every thread polls).  On a timeout
    //    the CTA records it and waits (bounded) once more for its copies
    //    before its shared memory is released.
    bool ok = false;
    const uint32_t first_cap = a.first_wait_polls < 0 ? DECODE_WAIT_LIMIT : (uint32_t)a.first_wait_polls;
    for (uint32_t i = 0; i < first_cap && !ok; ++i) ok = dec_try_wait(bar, 0);
    if (__syncthreads_or(!ok)) {
        if (tid == 0) {
            atomicExch(&g_device_error, DEV_TIMEOUT);
            for (uint32_t i = 0; i < DECODE_WAIT_LIMIT; ++i)
                if (dec_try_wait(bar, 0)) break;
            for (uint32_t i = 0; i < DECODE_WAIT_LIMIT; ++i)
                if (dec_try_wait(bar_ring, 0)) break;
        }
        return;
    }
    if (p < 0) {  // not a state this library wrote: record it, touch nothing
        if (tid == 0) {
            atomicExch(&g_device_error, DEV_BAD_POS);
            for (uint32_t i = 0; i < DECODE_WAIT_LIMIT; ++i)
                if (dec_try_wait(bar_ring, 0)) break;
        }
        return;
    }
    if (tid < D) {
        q_s[tid] = to_f32(tok[tid]);
        k_s[tid] = to_f32(tok[D + tid]);
        v_s[tid] = to_f32(tok[2 * D + tid]);
        gam_s[tid] = expf(log_sigmoid(to_f32(tok[3 * D + tid])));
    }
    __syncthreads();

    // 3. State update S <- diag(gamma) S + k^T v and readout q S, first (it
    //    needs only the token): the state's stores go out while the ring
    //    copies land and the window is scored.
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    const float4 vq = *reinterpret_cast<const float4 *>(v_s + j0 + cq * 4);
#pragma unroll
    for (int r = 0; r < RPT; ++r) {
        const int row = rg + r * RG;
        const float gi = gam_s[row], ki = k_s[row], qi = q_s[row];
        float4 s = s_reg[r];
        s.x = gi * s.x + ki * vq.x;
        s.y = gi * s.y + ki * vq.y;
        s.z = gi * s.z + ki * vq.z;
        s.w = gi * s.w + ki * vq.w;
        Sg[(size_t)row * (D / 4) + cq] = s;
        acc.x += qi * s.x;
        acc.y += qi * s.y;
        acc.z += qi * s.z;
        acc.w += qi * s.w;
    }

    // The ring copies (bounded wait; on a timeout the CTA records it and
    // waits once more before its shared memory is released).
    bool ok_ring = false;
    for (uint32_t i = 0; i < DECODE_WAIT_LIMIT && !ok_ring; ++i) ok_ring = dec_try_wait(bar_ring, 0);
    if (__syncthreads_or(!ok_ring)) {
        if (tid == 0) {
            atomicExch(&g_device_error, DEV_TIMEOUT);
            for (uint32_t i = 0; i < DECODE_WAIT_LIMIT; ++i)
                if (dec_try_wait(bar_ring, 0)) break;
        }
        return;
    }

    // 4. Window logits: history tokens p - nh .. p - 1 (ring slot token % w),
    //    the current token, then the m meta keys.  Thread `sub` of a key
    //    covers dims {64 e + 8 sub .. 64 e + 8 sub + 7}, so eight threads
    //    read a 128-byte run of the key.
    const int nh = (int)(p < (int64_t)(w - 1) ? p : (int64_t)(w - 1));
    const int n = nh + 1;
    const int64_t first = p - nh;
    {
        const int sub = tid % KT;
        float qd[DPT];
#pragma unroll
        for (int e = 0; e < DPT; ++e) qd[e] = q_s[(e / 8) * 64 + sub * 8 + e % 8];
        for (int c0 = 0; c0 < n + m; c0 += KPP) {
            const int c = c0 + tid / KT;
            float part = 0.f;
            if (c < n + m) {
                const T *kr = c < nh ? rk + (size_t)((first + c) % w) * D : mu + (size_t)(c - n) * D;
#pragma unroll
                for (int e0 = 0; e0 < DPT; e0 += 8) {
                    float x[8];
                    if (c == nh) {
#pragma unroll
                        for (int e = 0; e < 8; ++e) x[e] = k_s[(e0 / 8) * 64 + sub * 8 + e];
                    } else {
                        load8(kr + (e0 / 8) * 64 + sub * 8, x);
                    }
#pragma unroll
                    for (int e = 0; e < 8; ++e) part += qd[e0 + e] * x[e];
                }
            }
#pragma unroll
            for (int o = KT / 2; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
            if (c < n + m && sub == 0) sc[c] = part;
        }
    }
    __syncthreads();

    // 5. Softmax statistics over the window and the sinks; each logit is
    //    replaced by its exponential e^{s - M}, so that the anchor sum below
    //    takes every key's once instead of once per thread that uses it.
    if (warp == 0) {
        float M = -INFINITY;
        for (int c = lane; c < n + m; c += 32) M = fmaxf(M, sc[c]);
        M = warp_max(M);
        float Z = 0.f;
        for (int c = lane; c < n + m; c += 32) {
            const float e = expf(sc[c] - M);
            sc[c] = e;
            Z += e;
        }
        Z = warp_sum(Z);
        if (lane == 0) stat[1] = head_alpha(a.alpha_h, a.alpha, u % H) / Z;
    }
    __syncthreads();
    const float scale = stat[1];

    // 6. Anchor partial: this row group's share of the window keys, for this
    //    CTA's columns.
    for (int c = rg; c < n; c += RG) {
        const float pc = sc[c] * scale;
        const float4 vv = c < nh ? load4(rv + (size_t)((first + c) % w) * D + j0 + cq * 4)
                                 : *reinterpret_cast<const float4 *>(v_s + j0 + cq * 4);
        acc.x += pc * vv.x;
        acc.y += pc * vv.y;
        acc.z += pc * vv.z;
        acc.w += pc * vv.w;
    }

    *reinterpret_cast<float4 *>(red + rg * DH + cq * 4) = acc;

    // 7. Ring slot p % w takes this CTA's half of the current k and v (the
    //    slot held token p - w, which is outside this step's window).
    if (tid < DH) {
        const size_t slot = ((size_t)u * w + (size_t)(p % w)) * D + j0 + tid;
        static_cast<T *>(a.ring_k)[slot] = tok[D + j0 + tid];
        static_cast<T *>(a.ring_v)[slot] = tok[2 * D + j0 + tid];
    }
    __syncthreads();
    if (tid < DH) {
        float y = 0.f;
#pragma unroll 8
        for (int r = 0; r < RG; ++r) y += red[r * DH + tid];
        static_cast<T *>(a.y)[(size_t)u * D + j0 + tid] = from_f32<T>(y);
    }
}

}  // namespace lizard
