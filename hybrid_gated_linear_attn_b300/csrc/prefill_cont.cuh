// prefill_cont.cuh -- the start position of a prefill that continues a
// sequence.
//
// A prompt that continues a sequence (chunked prefill while serving, or a
// prompt after decoded tokens) starts from the recurrent state instead of
// zero -- S carries the whole past of the gate branch (Lizard,
// gist.science/de section 2 item 1, S_t = diag(sigmoid(g_t)) S_{t-1} +
// k_t^T v_t) -- and its first w-1 tokens see earlier tokens in their anchor
// window (item 2), which the state keeps in its ring (token p in slot p % w).
// Every CTA of sequence b needs p0 = pos[b], the position of the first new
// token, and the sequence ends at pos[b] = p0 + L.  The CTAs run in no fixed
// order, so the position is read and advanced in one atomic pass: each of
// the `ctas` CTAs of the sequence adds 2^40 to pos[b] and takes p0 from the
// low 40 bits of the value it got back; the CTA whose addition was the last
// (ctas - 1 earlier ones) writes p0 + L.  A pos outside [0, 2^40) before
// the call is seen by the first CTA (negative) or the last (too large) and
// reported (DEV_BAD_POS); p0 is then those low bits, so every access stays
// inside the caller's buffers although the results are undefined.
#pragma once

#include "common.cuh"

namespace lizard {

constexpr unsigned long long CONT_POS_TICK = 1ull << 40;

// One thread of each CTA of sequence b calls this once, at the start.
__device__ __forceinline__ int64_t take_start_position(int64_t *pos, int ctas, int L)
{
    unsigned long long *p = reinterpret_cast<unsigned long long *>(pos);
    const unsigned long long old = atomicAdd(p, CONT_POS_TICK);
    const long long cnt = (long long)old >> 40;
    const int64_t p0 = (int64_t)(old & (CONT_POS_TICK - 1));
    if (cnt < 0 || cnt >= ctas) atomicExch(&g_device_error, DEV_BAD_POS);
    else if (cnt == ctas - 1) atomicExch(p, (unsigned long long)(p0 + L));
    return p0;
}

// Source row of history token tau (-64 * nchunks <= tau < 0) for a CTA that
// reads the window history from the ring itself (it writes the ring only
// after reading it): ring slot (p0 + tau) % w, or null when the token is not
// in the window history (tau < -nvalid).
template <typename T>
__device__ __forceinline__ const T *history_row(const T *ring, int64_t p0, int tau, int nvalid, int w, int d)
{
    return tau < -nvalid ? nullptr : ring + (size_t)((p0 + tau) % w) * d;
}

}  // namespace lizard
