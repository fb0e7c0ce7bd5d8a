// prefill_cont.cuh -- inputs of a prefill that continues a sequence.
//
// A prompt that continues a sequence (chunked prefill while serving, or a
// prompt after decoded tokens) starts from the recurrent state instead of
// zero -- S carries the whole past of the gate branch (Lizard,
// gist.science/de section 2 item 1, S_t = diag(sigmoid(g_t)) S_{t-1} +
// k_t^T v_t) -- and its first w-1 tokens see earlier tokens in their anchor
// window (item 2), which the state keeps in its ring (token p in slot p % w).
//
// The prefill kernels write the state in place when they finish, and their
// CTAs run in no fixed order (the heads of one sequence share pos[b]; the
// segments of one sequence share S and the ring).  So before the prefill
// this kernel copies what the prefill reads from the state into scratch:
//   p0    [B]             pos[b], the position of the first new token
//   hist  [units][HR][d]  row HR - 1 - x holds token p0 - 1 - x for
//                         x < min(p0, w - 1), read from ring slot
//                         (p0 - 1 - x) % w; every other row is zero
// A pos outside [0, 2^40) is reported (DEV_BAD_POS) and read as 0, so that
// every access of the prefill stays inside the caller's buffers.
#pragma once

#include "common.cuh"

namespace lizard {

constexpr int64_t CONT_POS_LIMIT = (int64_t)1 << 40;
constexpr int CONT_THREADS = 256;

// grid = B * H (one CTA per unit); row16 = 16-byte words per token row.
__global__ void __launch_bounds__(CONT_THREADS) continue_prologue_kernel(
    const uint4 *ring_k, const uint4 *ring_v, const int64_t *pos, int H, int w, int HR, int row16,
    uint4 *hist_k, uint4 *hist_v, int64_t *p0_out)
{
    const int unit = blockIdx.x, b = unit / H, h = unit % H;
    int64_t p = pos[b];
    if (p < 0 || p >= CONT_POS_LIMIT) {
        if (h == 0 && threadIdx.x == 0) atomicExch(&g_device_error, DEV_BAD_POS);
        p = 0;
    }
    const int nvalid = (int)(p < (int64_t)(w - 1) ? p : (int64_t)(w - 1));
    const uint4 *rk = ring_k + (size_t)unit * w * row16, *rv = ring_v + (size_t)unit * w * row16;
    uint4 *hk = hist_k + (size_t)unit * HR * row16, *hv = hist_v + (size_t)unit * HR * row16;
    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
    for (int e = threadIdx.x; e < HR * row16; e += CONT_THREADS) {
        const int r = e / row16, x = e % row16;
        const int back = HR - r;  // this row holds token p - back
        uint4 kk = zero, vv = zero;
        if (back <= nvalid) {
            const size_t slot = (size_t)((p - back) % w);
            kk = rk[slot * row16 + x];
            vv = rv[slot * row16 + x];
        }
        hk[e] = kk;
        hv[e] = vv;
    }
    if (h == 0 && threadIdx.x == 0) p0_out[b] = p;
}

}  // namespace lizard
