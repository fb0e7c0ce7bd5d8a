// prefill_ws.cuh -- chunked Lizard prefill on tcgen05 tensor cores as a
// warp-specialised pipeline (bf16 inputs, d = 128 or 64, window w <= 129:
// a band of up to two earlier chunks).
//
// Operator: gated linear attention (Lizard, gist.science/de section 2 item 1)
// + anchor window with meta-memory sinks (item 2) + alpha combine (item 3).
// The chunked, log-space form follows the page's "Hardware-bewusster
// Algorithmus" section: cumulative gate terms are kept as log-space prefix
// sums and folded into the query/key operands, so the intra-chunk work is
// plain GEMMs on the tensor cores.
//
// One CTA walks the chunks (C = 64 tokens) of one (batch, head) sequence.
// Per chunk c (tokens c0 .. c0+63), with b_t = sum_{r=c0..t} log2 sigmoid(g_r)
// per key dim (fp32, base 2) and the reference r = b_{c0+31} (the end of the
// first half of the chunk):
//
//   SC  [t, s'] = q_t . k_s'  over the band (previous chunk, this chunk)
//                 and q_t . mu_j                              tcgen05, M=64
//   A   [t, s]  = QR_t . KR_s,  QR = q 2^{b-r}, KR = k 2^{r-b}  tcgen05, M=64
//   W   [t, s'] = alpha softmax-with-sinks(SC)[t, s'] + A[t, s] (s <= t)
//   Y^T [j, t]  = S16 QR^T + V_band^T W^T                       tcgen05, M=128
//                 (S16 = bf16(S_{c-1}^T diag(2^r)) in tensor memory)
//   S^T        <- S^T diag(2^{b_last}) + V^T KL,  KL = k 2^{b_last - b}
//
// The state is kept as Shat = S / F per key dim, F = 2^{b_last - r} of the
// last chunk folded in, because then the state update takes the same key
// operand as A:  KL = KR F, so  S_c / F_c = (S_{c-1} 2^r) + V^T KR  in the
// Shat form.  Per chunk the state pass scales Shat by F_{c-1} 2^{r_c} (which
// is also the scale of S16), and the final state is Shat F.  Only two
// operand tiles per chunk, so they are double-buffered and the gate prep of
// chunk c+1 runs while chunk c is in its softmax and output products.
//
// The factors of A have exponents within +-(half-chunk decay span); a chunk
// whose half-span exceeds SPAN2_MAX (base 2) for some key dimension is
// "unsafe": its A is computed exactly on the CUDA cores instead
// (sum_i q k 2^{b_t - b_s}, exponent <= 0), its QR uses r = 0, its key
// operand is KL itself and its F is 1.  So every gate value is handled.
//
// Warp roles (20 warps):
//   warp 0       TMA producer: q, k, v tiles (k/v ring of NP+2); L2 prefetch of g
//   warp 1       MMA issuer (one thread): window and meta scores SC
//   warp 2       MMA issuer (one thread): the two output products
//   warp 3       MMA issuer (one thread): intra-chunk scores A, the state update
//   warps 4-7    state pass (Shat scale, S16) and the y epilogue (one chunk
//                behind); the final state
//   warps 8-15   gate prep: log-sigmoid (g read into registers one chunk
//                ahead), prefix sums, the QR / KR operands and scale vectors
//   warps 16-19  window softmax: W from SC and A
// Every hand-off is an mbarrier; every wait is bounded (a timeout records
// DEV_TIMEOUT, drains the copies and products in flight, and returns).
//
// Head dim d = 64 runs on the same tiles, 128 wide: the key/value dims
// 64..127 of every shared-memory tile are zero (cleared at set-up; the TMA
// loads only the first 64-dim box), so the state's extra rows and columns
// stay zero.  Products over the key dim (scores, A, the readout) take d / 16
// K-steps; the gate prep and the state pass skip the padding.
#pragma once

#include "common.cuh"
#include "prefill_cont.cuh"
#include "sm100.cuh"

namespace lizard {
namespace ws {

using namespace sm100;

constexpr int C = 64;
constexpr int D = 128;
constexpr int NWARPS = 20;
constexpr int THREADS = NWARPS * 32;
constexpr int W_TMA = 0, W_MMA = 1, W_MMAY = 2, W_MMAS = 3, W_EPI = 4, W_PREP = 8, W_SOFT = 16;
constexpr int EPI_N = 128, PREP_N = 256, SOFT_N = 128;
enum : int { NB_EPI = 1, NB_PREP = 2, NB_SOFT = 3, NB_EPI_R = 4, NB_PREP_R = 5, NB_SOFT_R = 6 };
constexpr int META_ROWS = 16;
constexpr int KROWS = C + META_ROWS;       // key tile rows: 64 tokens, then the meta keys
constexpr float LOG2E = 1.4426950408889634f;
constexpr float SPAN2_MAX = 100.f;         // half-chunk decay span limit (base 2) of the GEMM path
constexpr uint32_t WAIT_LIMIT = 1u << 21;

// Shared memory (offsets from a 1024-aligned base).
constexpr uint32_t KB_K = KROWS * 128;     // one 64-dim block of a key tile (80 rows)
constexpr uint32_t KB_T = C * 128;         // one 64-dim block of a 64-row tile
constexpr uint32_t SLOT = 2 * KB_K + 2 * KB_T;
constexpr uint32_t SLOT_V = 2 * KB_K;      // v tile within a slot
constexpr uint32_t OPB = 4 * KB_T;         // one operand buffer: QR tile, then KR tile
constexpr int NVEC = 3;                    // per operand buffer: sig, tau, F (fp32 [128] each)
// A band of NP earlier chunks.  NP <= 1: a k/v ring of NP + 2 slots (one
// loads ahead) and two q stages.  NP = 2 (windows 66 .. 129): three slots
// and one q stage, to fit shared memory.
template <int NP>
struct Smem {
    static constexpr int NR = NP == 2 ? 3 : NP + 2;
    static constexpr int QS = NP == 2 ? 1 : 2;    // q stages
    static constexpr uint32_t KV = 0;
    static constexpr uint32_t Q = KV + NR * SLOT;
    static constexpr uint32_t OP = Q + QS * 2 * KB_T;      // two operand buffers
    static constexpr uint32_t W = OP + 2 * OPB;
    static constexpr uint32_t VEC = W + (NP + 1) * KB_T;   // [2][NVEC][128], then tot[4][128] (fp32)
    static constexpr uint32_t FLAG = VEC + (2 * NVEC * 128 + 4 * 128) * 4;  // unsafe[2], abort
    static constexpr uint32_t BAR = FLAG + 16;
    static constexpr int NBAR = 2 * QS + 4 * NR + 4 + 14;
    static constexpr uint32_t TSLOT = BAR + NBAR * 8;
    static constexpr uint32_t USED = TSLOT + 16;
    static constexpr uint32_t BYTES = USED + 1024;
    static_assert(BYTES <= 232448, "shared memory budget");
};

// Tensor-memory columns (512 allocated).
constexpr uint32_t T_S = 0, T_S16 = 128, T_Y = 192, T_SC = 256;
// With NP = 2 the intra-chunk scores A reuse the current chunk's score
// columns: the A product waits until the softmax has read them.
template <int NP>
struct Tmem {
    static constexpr uint32_t SC_COLS = 64 * NP + 64 + META_ROWS;
    static constexpr uint32_t A = NP == 2 ? T_SC + 64 * NP : T_SC + SC_COLS;
    static_assert(A + 64 <= 512 && T_SC + SC_COLS <= 512, "tensor memory budget");
};

struct WsArgs {
    const __nv_bfloat16 *g, *mu, *k, *v;
    __nv_bfloat16 *y;
    float *S_out;
    __nv_bfloat16 *ring_k, *ring_v;
    int64_t *pos;
    float alpha;
    int H, L, w, m;
    // Sequence segments: CTA (unit, seg) covers chunks [seg*seg_chunks,
    // (seg+1)*seg_chunks) and starts from S_init[unit][seg-1] (row = key
    // dim), the state after the earlier segments; segment 0 starts from S0.
    const float *S_init;
    int seg_chunks, nseg;
    // Continuation of a sequence (0 / null for a prompt from the empty
    // state): with cont = 1 every CTA takes the start position from pos
    // (take_start_position) and the first segment sees the window history
    // as chunk -1: from `hist` ([units][2][64][d], keys then values, row r =
    // token r - 64, zero where no key) when given, else from the ring, which
    // the CTA then writes only at its end (one segment).  S0 [units][d][d] is
    // the start state of the first segment (may be S_out when there is one
    // segment: it is read before S_out is written).
    int cont;
    const float *S0;
    const __nv_bfloat16 *hist;
    const float *alpha_h;  // per-head anchor weights (null: alpha)
    int group;             // query heads per key/value head (tk, tv map B x H / group heads)
};

// Optional clock trace of CTA 0 (compiled with -DLIZARD_TRACE): one clock64
// stamp per (chunk, event), read by lizard_debug_trace.
#ifdef LIZARD_TRACE
constexpr int TRACE_CHUNKS = 64, TRACE_EVENTS = 32;
__device__ unsigned long long g_ws_trace[TRACE_CHUNKS][TRACE_EVENTS];
#define LZ_TRACE(pc, ev)                                                              \
    do {                                                                              \
        if (blockIdx.x == 0 && (threadIdx.x & 31) == 0 && (pc) < TRACE_CHUNKS && (ev) < TRACE_EVENTS) g_ws_trace[(pc)][(ev)] = clock64(); \
    } while (0)
#else
#define LZ_TRACE(pc, ev) \
    do {                 \
    } while (0)
#endif

// ---------------------------------------------------------------- helpers
__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// log2(sigmoid(g)) = min(g, 0) log2(e) - log2(1 + u),  u = 2^{-|g| log2(e)} in (0, 1];
// log2(1 + u) = u P(u) with a degree-7 least-squares polynomial (absolute
// error < 4e-7, exactly 0 at u = 0 so open gates give no decay).
__device__ __forceinline__ float log2_sigmoid(float g)
{
    const float u = ex2(-fabsf(g) * LOG2E);
    float p = 0.015127916f;
    p = fmaf(p, u, -0.078158207f);
    p = fmaf(p, u, 0.19238505f);
    p = fmaf(p, u, -0.32461637f);
    p = fmaf(p, u, 0.47311336f);
    p = fmaf(p, u, -0.72051549f);
    p = fmaf(p, u, 1.4426640f);
    return fminf(g, 0.f) * LOG2E - u * p;
}
// Packed fp32x2 arithmetic (one instruction for a pair of key dims).
__device__ __forceinline__ uint64_t pk2(float2 a)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a.x), "f"(a.y));
    return r;
}
__device__ __forceinline__ float2 upk2(uint64_t r)
{
    float2 a;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a.x), "=f"(a.y) : "l"(r));
    return a;
}
__device__ __forceinline__ float2 add2(float2 a, float2 b)
{
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(pk2(a)), "l"(pk2(b)));
    return upk2(r);
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b)
{
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(pk2(a)), "l"(pk2(b)));
    return upk2(r);
}
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c)
{
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(pk2(a)), "l"(pk2(b)), "l"(pk2(c)));
    return upk2(r);
}
// log2_sigmoid of a pair: min(g, 0) log2(e) - log2(1 + 2^{-|g| log2(e)}),
// both transcendentals on the MUFU pipe (short dependency chain).
__device__ __forceinline__ float lg2(float x)
{
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float rcp(float x)
{
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float2 log2_sigmoid2(float2 g)
{
    const float ua = ex2(-fabsf(g.x) * LOG2E), ub = ex2(-fabsf(g.y) * LOG2E);
    return make_float2(fminf(g.x, 0.f) * LOG2E - lg2(1.f + ua), fminf(g.y, 0.f) * LOG2E - lg2(1.f + ub));
}
__device__ __forceinline__ float2 bf2_to_f2(uint32_t u)
{
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u));
}
__device__ __forceinline__ uint32_t f2_to_bf2(float lo, float hi)
{
    __nv_bfloat162 r = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&r);
}
// Streaming 4-byte load (read once: no L1 allocation).
__device__ __forceinline__ uint32_t ld_stream_u32(const void *p)
{
    uint32_t r;
    asm volatile("ld.global.nc.L1::no_allocate.b32 %0, [%1];" : "=r"(r) : "l"(p));
    return r;
}
// Bulk prefetch of `bytes` (a multiple of 16, 16-byte aligned) into L2.
__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}
__device__ __forceinline__ uint32_t tlane(uint32_t quarter) { return (32u * quarter) << 16; }
__device__ __forceinline__ void named_bar(int id, int n) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory"); }
__device__ __forceinline__ bool named_bar_and(int id, int n, bool p)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred pi, po;\n\t"
        "setp.ne.u32 pi, %1, 0;\n\t"
        "bar.red.and.pred po, %2, %3, pi;\n\t"
        "selp.u32 %0, 1, 0, po;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)p), "r"(id), "r"(n)
        : "memory");
    return r != 0;
}
__device__ __forceinline__ bool named_bar_or(int id, int n, bool p)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred pi, po;\n\t"
        "setp.ne.u32 pi, %1, 0;\n\t"
        "bar.red.or.pred po, %2, %3, pi;\n\t"
        "selp.u32 %0, 1, 0, po;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)p), "r"(id), "r"(n)
        : "memory");
    return r != 0;
}
// A role-wide wait: lane 0 of the role's first warp polls the mbarriers
// (`poll`), the role's other warps block in a named barrier meanwhile, so a
// waiting role takes no issue slots.  The AND-reduction barrier hands every
// thread the same verdict.  Readers of data produced by the async proxy or
// the tensor cores are ordered after the poller's acquire by this barrier
// (and by tcgen05.fence::after_thread_sync for tensor memory).
template <typename Poll>
__device__ __forceinline__ bool role_wait(bool leader_warp, int lane, int id, int n, Poll poll)
{
    bool ok = true;
    if (leader_warp) {
        if (lane == 0) ok = poll();
        __syncwarp();
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    }
    return named_bar_and(id, n, ok);
}
// Bounded wait on phase `use` (its parity) of an mbarrier; false on timeout
// or when another role already gave up.
__device__ __forceinline__ bool bwait(uint64_t *bar, uint32_t use, volatile int *abort_flag)
{
    const uint32_t a = smem_u32(bar), par = use & 1u;
#pragma unroll 1
    for (uint32_t i = 0; i < WAIT_LIMIT / 256u; ++i) {
        uint32_t ok;
        // up to 256 polls in one loop of the PTX itself (small code)
        asm volatile(
            "{\n\t.reg .pred p;\n\t.reg .u32 n;\n\t"
            "mov.u32 n, 256;\n\t"
            "LZ_POLL_%=:\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "@p bra.uni LZ_DONE_%=;\n\t"
            "sub.u32 n, n, 1;\n\t"
            "setp.ne.u32 p, n, 0;\n\t"
            "@p bra.uni LZ_POLL_%=;\n\t"
            "LZ_DONE_%=:\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(a), "r"(par)
            : "memory");
        // p is true on success; after 256 failed polls n = 0 and p is false
        if (ok) return true;
        if (*abort_flag) return false;
    }
    return false;
}

// One product D (+)= A B^T of bf16 tiles in shared memory, K = 16 * nk.
// Both operand descriptors advance by (step_a, step_b) bytes per k-step and
// by (blk_a, blk_b) bytes after every fourth step (next 64-wide block of a
// 128-byte-swizzled K-major tile).  A rolled loop keeps the issuing code
// small: the instruction cache is shared by every role of the CTA.
__device__ __forceinline__ void mma_chain(uint32_t d, uint64_t da, uint64_t db, uint32_t idesc, uint32_t acc, int nk,
                                          uint32_t step_a, uint32_t step_b, uint32_t blk_a, uint32_t blk_b)
{
#pragma unroll 1
    for (int kk = 0; kk < nk; ++kk) {
        const uint32_t oa = ((kk >> 2) * blk_a + (kk & 3) * step_a) >> 4, ob = ((kk >> 2) * blk_b + (kk & 3) * step_b) >> 4;
        mma_bf16_ss(d, da + oa, db + ob, idesc, acc | (uint32_t)(kk > 0));
    }
}

// FAST: the window fits one 64-slot overlay (NP = 1, w <= 64): only that
// softmax is compiled in, which keeps the chunk loop's code small.  W64
// (with FAST): w = 64 and a prompt from the empty state, so that every slot
// of the overlay is a key of its row -- in the first chunk the missing
// earlier chunk's score columns hold -inf -- and the masked selection is
// left out as well.
template <int NP, int DH, bool FAST = false, bool W64 = false>
__global__ void __launch_bounds__(THREADS, 1)
    prefill_ws_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                      const __grid_constant__ CUtensorMap tv, const WsArgs a)
{
    using SM = Smem<NP>;
    using TM = Tmem<NP>;
    constexpr int NR = SM::NR, QS = SM::QS;
    constexpr int NB = NP + 1;  // band chunks
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = smem_align1024(smem_raw);
    const uint32_t sb = smem_u32(sm);
    // Scale vectors of operand buffer b: vec + b * NVEC * 128 -> sig (state
    // pass: Shat scale), tau (S16 scale), F (the chunk's state factor).
    float *vec = reinterpret_cast<float *>(sm + SM::VEC);
    float *tot = vec + 2 * NVEC * 128;                          // [4][128] quarter totals
    volatile int *unsafe_f = reinterpret_cast<volatile int *>(sm + SM::FLAG);  // [2], per operand buffer
    volatile int *abort_f = unsafe_f + 2;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + SM::BAR);
    // k and v of a slot load and free separately: a key tile is free once
    // the band scores that read it are done, a value tile after its state
    // update and the output products (two arrivals).
    uint64_t *q_full = bars, *q_empty = bars + QS, *k_full = bars + 2 * QS, *k_empty = k_full + NR;
    uint64_t *v_full = k_empty + NR, *v_empty = v_full + NR;
    uint64_t *op_full = v_empty + NR, *op_free = op_full + 2;   // per operand buffer
    uint64_t *sc_full = op_free + 2, *a_full = sc_full + 1, *sc_free = sc_full + 2, *w_full = sc_full + 3,
             *w_free = sc_full + 4, *s_ready = sc_full + 5, *st_done = sc_full + 6, *s16_free = sc_full + 7,
             *y_full = sc_full + 8, *y_free = sc_full + 9, *drain = sc_full + 10, *drain_y = sc_full + 11,
             *drain_s = sc_full + 12, *sc_read = sc_full + 13;  // sc_read: NP = 2 only
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + SM::TSLOT);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nseg = a.nseg;
    const int unit = blockIdx.x / nseg, seg = blockIdx.x % nseg, h = unit % a.H;
    const int L = a.L, w = a.w, m = a.m;
    constexpr int d = DH, nbox = d / 64, nk = d / 16;  // head dim; 64-dim boxes per tile, K-steps over the key dim
    const int nchunks = (L + C - 1) / C;
    // This CTA's chunks, and the first chunk it loads: the band of its first
    // chunk reaches NP chunks back into the previous segment, or into the
    // window history (chunk -1) when the prompt continues a sequence.
    const int c_begin = seg * a.seg_chunks, c_end = min(nchunks, c_begin + a.seg_chunks);
    const int c_lo = c_begin > 0 || a.cont ? c_begin - NP : 0;
    const bool last_seg = seg == nseg - 1;
    int64_t *p0_slot = reinterpret_cast<int64_t *>(sm + SM::TSLOT + 8);

    // ---------------------------------------------------------- set-up
    if (warp == W_MMA) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int i = 0; i < QS; ++i) {
            mbar_init(&q_full[i], 1);
            mbar_init(&q_empty[i], 2);   // scores issued + prep read q
        }
        for (int i = 0; i < NR; ++i) {
            mbar_init(&k_full[i], 1);
            mbar_init(&k_empty[i], 2);   // band scores + prep read the raw keys
            mbar_init(&v_full[i], 1);
            mbar_init(&v_empty[i], 2);   // state update + output products
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&op_full[i], 1);
            mbar_init(&op_free[i], 2);   // A + state update, the readout
        }
        for (int i = 0; i < 14; ++i) mbar_init(&sc_full[i], 1);
        unsafe_f[0] = 0;
        unsafe_f[1] = 0;
        *abort_f = 0;
        fence_mbar_init();
        prefetch_tmap(&tq);
        prefetch_tmap(&tk);
        prefetch_tmap(&tv);
        *p0_slot = a.cont ? take_start_position(a.pos + unit / a.H, a.H * nseg, L) : 0;
    }
    if (a.cont) __syncthreads();  // p0
    // Start position (0 for a prompt from the empty state; read from shared
    // memory only after the barrier above), and the history tokens
    // -nvalid .. -1 in the window.
    const int64_t p0 = a.cont ? *p0_slot : 0;
    const int kvu = kv_unit(unit, a.H, a.group);  // this head's key/value head
    const int nvalid = a.cont ? (int)min(p0, (int64_t)(w - 1)) : 0;
    if constexpr (d < D) {
        // the padding dims of the k/v ring, the q stages and the operand buffers
        for (uint32_t e = tid; e < SM::W / 16; e += THREADS)
            *reinterpret_cast<uint4 *>(sm + 16 * e) = make_uint4(0u, 0u, 0u, 0u);
        __syncthreads();
    }
    if (c_lo < 0) {
        // Window history (chunks c_lo .. -1) into k/v slots 0 .. -c_lo - 1,
        // zero rows where no key, in the swizzled layout of a TMA-loaded
        // tile.  (`hist` holds chunk -1 only: one earlier chunk.)
        const __nv_bfloat16 *rk = a.ring_k + (size_t)unit * w * d, *rv = a.ring_v + (size_t)unit * w * d;
        const __nv_bfloat16 *hk = a.hist ? a.hist + (size_t)unit * 2 * C * d : nullptr;
        const __nv_bfloat16 *hv = a.hist ? hk + C * d : nullptr;
        const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
        for (int e = tid; e < -c_lo * C * (d / 8); e += THREADS) {
            const int cc = e / (C * (d / 8)), r = (e / (d / 8)) % C, i8 = (e % (d / 8)) * 8;
            const int tau = (c_lo + cc) * C + r;  // token position relative to the first new one
            const __nv_bfloat16 *kr = hk ? hk + (size_t)r * d : history_row(rk, p0, tau, nvalid, w, d);
            const __nv_bfloat16 *vr = hk ? hv + (size_t)r * d : history_row(rv, p0, tau, nvalid, w, d);
            const uint32_t sw = sw128_offset(r, (i8 % 64) * 2);
            uint8_t *slot = sm + SM::KV + cc * SLOT;
            *reinterpret_cast<uint4 *>(slot + (i8 / 64) * KB_K + sw) = kr ? *reinterpret_cast<const uint4 *>(kr + i8) : zero;
            *reinterpret_cast<uint4 *>(slot + SLOT_V + (i8 / 64) * KB_T + sw) =
                vr ? *reinterpret_cast<const uint4 *>(vr + i8) : zero;
        }
    }
    // Meta keys of this head into rows 64..79 of every key tile (zero past m).
    for (int e = tid; e < NR * META_ROWS * 64; e += THREADS) {
        const int s = e / (META_ROWS * 64), rem = e % (META_ROWS * 64), r = rem / 64, ip = rem % 64;
        const int i = 2 * ip;
        uint32_t val = 0u;
        if (r < m && i < d) val = *reinterpret_cast<const uint32_t *>(a.mu + ((size_t)h * m + r) * d + i);
        *reinterpret_cast<uint32_t *>(sm + SM::KV + s * SLOT + (i / 64) * KB_K +
                                      sw128_offset(C + r, (i % 64) * 2)) = val;
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // The band chunks before this CTA's first chunk (slots 0 .. c_begin -
    // c_lo - 1, first use): loaded, or the window history in place.
    auto preband_ready = [&](uint64_t *full) {
        for (int i = 0; i < c_begin - c_lo; ++i)
            if (!bwait(&full[i], 0, abort_f)) return false;
        return true;
    };
    bool failed = false;
    auto give_up = [&]() {
        failed = true;
        *abort_f = 1;
        atomicExch(&g_device_error, DEV_TIMEOUT);
    };


    if (warp == W_TMA) {
        // ------------------------------------------------------ producer
        if (lane == 0) {
            uint32_t k_issued[NR] = {}, v_issued[NR] = {}, q_issued[QS] = {};
            // The gate logits go straight to registers in the prep role; a
            // bulk prefetch two chunks ahead keeps them in L2.
            auto prefetch_g = [&](int c) {
                const int n = min(C, L - c * C);
                prefetch_l2(a.g + ((size_t)unit * L + (size_t)c * C) * d, (uint32_t)n * d * 2u);
            };
            for (int c = c_begin; c < min(c_end, c_begin + 2); ++c) prefetch_g(c);
            // One 64-token tile: nbox boxes of 64 dims, `blk` bytes apart.
            auto load_tile = [&](uint8_t *dst, uint32_t blk, const CUtensorMap *map, uint64_t *bar, int c, int u) {
                mbar_arrive_expect_tx(bar, nbox * KB_T);
                for (int x = 0; x < nbox; ++x) tma_load_3d(dst + x * blk, map, bar, 64 * x, c * C, u);
            };
            // keys and values of the band chunks before this segment; the
            // window history (chunk -1) is in place since the set-up
            for (int c = c_lo; c < c_begin; ++c) {
                const int s = (c - c_lo) % NR;
                uint8_t *base = sm + SM::KV + s * SLOT;
                if (c < 0) {
                    mbar_arrive(&k_full[s]);
                    mbar_arrive(&v_full[s]);
                } else {
                    load_tile(base, KB_K, &tk, &k_full[s], c, kvu);
                    load_tile(base + SLOT_V, KB_T, &tv, &v_full[s], c, kvu);
                }
                ++k_issued[s];
                ++v_issued[s];
            }
            for (int c = c_begin; c < c_end && !failed; ++c) {
                const int pc = c - c_begin, r = c - c_lo;
                if (c + 2 < c_end) prefetch_g(c + 2);
                const int s = r % NR;
                uint8_t *base = sm + SM::KV + s * SLOT;
                if (r >= NR && !bwait(&k_empty[s], r / NR - 1, abort_f)) { give_up(); break; }
                load_tile(base, KB_K, &tk, &k_full[s], c, kvu);
                ++k_issued[s];
                LZ_TRACE(pc, 15);
                const int qs = pc % QS;
                if (pc >= QS && !bwait(&q_empty[qs], pc / QS - 1, abort_f)) { give_up(); break; }
                load_tile(sm + SM::Q + qs * 2 * KB_T, KB_T, &tq, &q_full[qs], c, unit);
                ++q_issued[qs];
                LZ_TRACE(pc, 16);
                if (r >= NR && !bwait(&v_empty[s], r / NR - 1, abort_f)) { give_up(); break; }
                load_tile(base + SLOT_V, KB_T, &tv, &v_full[s], c, kvu);
                ++v_issued[s];
                LZ_TRACE(pc, 17);
            }
            // Drain: every copy issued has landed before shared memory is released.
            for (int s = 0; s < NR; ++s) {
                if (k_issued[s]) bwait(&k_full[s], k_issued[s] - 1, abort_f);
                if (v_issued[s]) bwait(&v_full[s], v_issued[s] - 1, abort_f);
            }
            for (int s = 0; s < QS; ++s)
                if (q_issued[s]) bwait(&q_full[s], q_issued[s] - 1, abort_f);
        }
        __syncwarp();
    } else if (warp == W_MMA) {
        // ------------------------------------------------------ MMA issuer: scores SC
        if (lane == 0) {
            const uint32_t id_sc_prev = instr_desc(64, 64, FMT_BF16, 0, 0);
            const uint32_t id_sc_cur = instr_desc(64, 64 + META_ROWS, FMT_BF16, 0, 0);
            for (int c = c_begin; c < c_end; ++c) {
                const int pc = c - c_begin, r = c - c_lo;
                const int s = r % NR, qs = pc % QS;
                const uint32_t qb = sb + SM::Q + qs * 2 * KB_T;
                if ((pc == 0 && !preband_ready(k_full)) ||
                    !bwait(&k_full[s], r / NR, abort_f) || !bwait(&q_full[qs], pc / QS, abort_f) ||
                    (pc >= 1 && !bwait(sc_free, pc - 1, abort_f))) { give_up(); break; }
                LZ_TRACE(pc, 24);
                tc_fence_after();
                // window + meta logits
#pragma unroll 1
                for (int j = 0; j <= NP; ++j) {
                    const int cj = c - NP + j;
                    if (cj < c_lo) continue;
                    const uint32_t kb = sb + SM::KV + ((cj - c_lo) % NR) * SLOT;
                    mma_chain(tmem + T_SC + 64 * j, smem_desc(qb, 16, 1024), smem_desc(kb, 16, 1024),
                              j == NP ? id_sc_cur : id_sc_prev, 0u, nk, 32, 32, KB_T, KB_K);
                }
                mma_commit(sc_full);
                mma_commit(&q_empty[qs]);
                LZ_TRACE(pc, 3);
                // The key tile of chunk c - NP: its last band scores are issued.
                if (c - NP >= c_lo) mma_commit(&k_empty[(c - NP - c_lo) % NR]);
            }
            // Drain: every product issued has completed before tensor memory is released.
            mma_commit(drain);
            bwait(drain, 0, abort_f);
        }
        __syncwarp();
    } else if (warp == W_MMAS) {
        // ------------------------------------------------------ MMA issuer: intra-chunk scores A, state update
        if (lane == 0) {
            const uint32_t id_st = instr_desc(128, 128, FMT_BF16, 1, 1);
            const uint32_t id_a = instr_desc(64, 64, FMT_BF16, 0, 0);
            // band chunks before the segment get no state update and no prep
            for (int c = c_lo; c < c_begin; ++c) {
                mbar_arrive(&v_empty[(c - c_lo) % NR]);
                mbar_arrive(&k_empty[(c - c_lo) % NR]);
            }
            for (int c = c_begin; c < c_end; ++c) {
                const int pc = c - c_begin, r = c - c_lo, s = r % NR, b = pc & 1;
                // intra-chunk decayed scores A (the A columns are free once the
                // previous chunk's softmax has read them)
                if (!bwait(&op_full[b], pc >> 1, abort_f) ||
                    (NP == 2 ? !bwait(sc_read, pc, abort_f) : (pc >= 1 && !bwait(sc_free, pc - 1, abort_f)))) {
                    give_up();
                    break;
                }
                LZ_TRACE(pc, 28);
                tc_fence_after();
                if (!unsafe_f[b]) {
                    const uint32_t ob = sb + SM::OP + b * OPB;
                    mma_chain(tmem + TM::A, smem_desc(ob, 16, 1024), smem_desc(ob + 2 * KB_T, 16, 1024), id_a, 0u, nk,
                              32, 32, KB_T, KB_T);
                    mma_commit(a_full);
                } else {
                    mbar_arrive(a_full);  // exact A, stored by the prep role before op_full
                }
                LZ_TRACE(pc, 4);
                mbar_arrive(&k_empty[s]);  // the prep of this chunk has read its raw keys
                if (!bwait(s_ready, pc, abort_f) || !bwait(&v_full[s], r / NR, abort_f)) { give_up(); break; }
                LZ_TRACE(pc, 26);
                tc_fence_after();
                // Shat^T += V^T K, K = KR (KL for an unsafe chunk)
                const uint32_t vb = sb + SM::KV + s * SLOT + SLOT_V, kb = sb + SM::OP + b * OPB + 2 * KB_T;
                mma_chain(tmem + T_S, smem_desc(vb, KB_T, 1024), smem_desc(kb, KB_T, 1024), id_st, 1u, 4, 2048, 2048, 0,
                          0);
                mma_commit(st_done);
                mma_commit(&op_free[b]);
                mma_commit(&v_empty[s]);
                LZ_TRACE(pc, 5);
            }
            mma_commit(drain_s);
            bwait(drain_s, 0, abort_f);
        }
        __syncwarp();
    } else if (warp == W_MMAY) {
        // ------------------------------------------------------ MMA issuer: outputs
        if (lane == 0) {
            const uint32_t id_y1 = instr_desc(128, 64, FMT_BF16, 0, 0);
            const uint32_t id_y2 = instr_desc(128, 64, FMT_BF16, 1, 0);
            for (int c = c_begin; c < c_end; ++c) {
                const int pc = c - c_begin, r = c - c_lo, b = pc & 1;
                // y^T = S16 QR^T (inter-chunk readout)
                if (!bwait(&op_full[b], pc >> 1, abort_f) || !bwait(s_ready, pc, abort_f) ||
                    (pc >= 1 && !bwait(y_free, pc - 1, abort_f))) { give_up(); break; }
                LZ_TRACE(pc, 27);
                tc_fence_after();
                const uint32_t ob = sb + SM::OP + b * OPB;
                {
                    const uint64_t dq = smem_desc(ob, 16, 1024);
#pragma unroll 1
                    for (int kk = 0; kk < nk; ++kk)
                        mma_bf16_ts(tmem + T_Y, tmem + T_S16 + kk * 8, dq + ((((kk >> 2) * KB_T) + (kk & 3) * 32) >> 4),
                                    id_y1, kk > 0);
                }
                mma_commit(s16_free);
                mma_commit(&op_free[b]);
                LZ_TRACE(pc, 6);
                // y^T += V_band^T W^T
                if (!bwait(w_full, pc, abort_f) || !bwait(&v_full[r % NR], r / NR, abort_f) ||
                    (pc == 0 && !preband_ready(v_full))) { give_up(); break; }
                LZ_TRACE(pc, 25);
                tc_fence_after();
#pragma unroll 1
                for (int j = 0; j <= NP; ++j) {
                    const int cj = c - NP + j;
                    if (cj < c_lo) continue;
                    const uint32_t vb = sb + SM::KV + ((cj - c_lo) % NR) * SLOT + SLOT_V;
                    mma_chain(tmem + T_Y, smem_desc(vb, KB_T, 1024), smem_desc(sb + SM::W + j * KB_T, 16, 1024), id_y2,
                              1u, 4, 2048, 32, 0, 0);
                }
                mma_commit(y_full);
                mma_commit(w_free);
                LZ_TRACE(pc, 7);
                // The value tile of chunk c - NP has no reader left among the
                // output products (its state update commits separately).
                if (c - NP >= c_lo) mma_commit(&v_empty[(c - NP - c_lo) % NR]);
            }
            mma_commit(drain_y);
            bwait(drain_y, 0, abort_f);
        }
        __syncwarp();
    } else if (warp >= W_EPI && warp < W_EPI + 4) {
        // ------------------------------------------------------ state pass + epilogue
        const int quarter = warp & 3;
        const int j = 32 * quarter + lane;  // value dim = tensor-memory lane
        const uint32_t tl = tmem + tlane(quarter);
        const bool live = j < d;            // lanes past d_v hold the zero padding: no stores
        {
            // Initial state: the state after the earlier segments, or S0
            // (zero when not given) for the first segment; zero padding.
            const float *Si = !live ? nullptr
                              : seg > 0 ? (a.S_init ? a.S_init + ((size_t)unit * (nseg - 1) + seg - 1) * d * d + j
                                                    : nullptr)
                                        : (a.S0 ? a.S0 + (size_t)unit * d * d + j : nullptr);
#pragma unroll 1
            for (int cc = 0; cc < D; cc += 16) {
                uint32_t z[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) z[e] = Si && cc + e < d ? __float_as_uint(Si[(size_t)(cc + e) * d]) : 0u;
                tmem_st16(tl + T_S + cc, z);
            }
            tmem_wait_st();
        }
        const int et = tid - W_EPI * 32;
        // y rows of chunk c_begin + py: read the accumulator, store bf16.
        auto epilogue = [&](int py) -> bool {
            if (!role_wait(warp == W_EPI, lane, NB_EPI_R, EPI_N, [&] { return bwait(y_full, py, abort_f); }))
                return false;
            LZ_TRACE(py, 10);
            tc_fence_after();
            const int c0 = (c_begin + py) * C, n = min(C, L - c0);
            __nv_bfloat16 *yp = a.y + ((size_t)unit * L + c0) * d + j;
            uint32_t r[4][16];
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) tmem_ld16(tl + T_Y + 16 * q4, r[q4]);
            tmem_wait_ld();
            // the accumulator is read: the next chunk's products may start
            tc_fence_before();
            named_bar(NB_EPI, EPI_N);
            if (et == 0) mbar_arrive(y_free);
            // Lanes j, j^1 trade halves of a token pair, so that each stores
            // two adjacent value dims of one token (4-byte stores): the even
            // lane token t, the odd lane token t + 1.
            const bool odd = lane & 1;
            __nv_bfloat16 *yq = yp - (odd ? 1 : 0) + (odd ? d : 0);
            const int t_odd = odd ? 1 : 0;
            uint32_t pk[4][8];
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4)
#pragma unroll
                for (int e = 0; e < 16; e += 2)
                    pk[q4][e / 2] = f2_to_bf2(__uint_as_float(r[q4][e]), __uint_as_float(r[q4][e + 1]));
            // rolled over the four 16-token groups: pk shifts down by one
            // group per pass (static register indices)
#pragma unroll 1
            for (int q4 = 0; q4 < 4; ++q4) {
#pragma unroll
                for (int e = 0; e < 16; e += 2) {
                    const uint32_t mine = pk[0][e / 2];
                    const uint32_t other = __shfl_xor_sync(0xffffffffu, mine, 1);
                    // even: (mine.lo, other.lo); odd: (other.hi, mine.hi)
                    const uint32_t out = odd ? __byte_perm(other, mine, 0x7632) : __byte_perm(mine, other, 0x5410);
                    if (live && 16 * q4 + e + t_odd < n)
                        *reinterpret_cast<uint32_t *>(yq + (size_t)(16 * q4 + e) * d) = out;
                }
#pragma unroll
                for (int g4 = 0; g4 < 3; ++g4)
#pragma unroll
                    for (int e = 0; e < 8; ++e) pk[g4][e] = pk[g4 + 1][e];
            }
            LZ_TRACE(py, 11);
            return true;
        };
        for (int c = c_begin; c < c_end; ++c) {
            const int pc = c - c_begin, b = pc & 1;
            if (!role_wait(warp == W_EPI, lane, NB_EPI_R, EPI_N, [&] {
                    return (pc == 0 || (bwait(st_done, pc - 1, abort_f) && bwait(s16_free, pc - 1, abort_f))) &&
                           bwait(&op_full[b], pc >> 1, abort_f);
                })) { give_up(); break; }
            LZ_TRACE(pc, 8);
            tc_fence_after();
            const float *sg = vec + b * NVEC * 128, *tv = sg + 128;
            // Shat <- Shat sig and S16 = bf16(Shat tau); sig = tau except in
            // an unsafe chunk, so one product serves both.
            const bool one = !unsafe_f[b];
#pragma unroll 1
            for (int cb = 0; cb < d; cb += 32) {
                uint32_t r0[16], r1[16];
                tmem_ld16(tl + T_S + cb, r0);
                tmem_ld16(tl + T_S + cb + 16, r1);
                tmem_wait_ld();
                uint32_t p16[16];
                if (one) {
#pragma unroll
                    for (int e = 0; e < 16; e += 2) {
                        const float2 sv = *reinterpret_cast<const float2 *>(sg + cb + e);
                        const float2 sw = *reinterpret_cast<const float2 *>(sg + cb + 16 + e);
                        const float2 a0 = mul2(make_float2(__uint_as_float(r0[e]), __uint_as_float(r0[e + 1])), sv);
                        const float2 a1 = mul2(make_float2(__uint_as_float(r1[e]), __uint_as_float(r1[e + 1])), sw);
                        r0[e] = __float_as_uint(a0.x);
                        r0[e + 1] = __float_as_uint(a0.y);
                        r1[e] = __float_as_uint(a1.x);
                        r1[e + 1] = __float_as_uint(a1.y);
                        p16[e / 2] = f2_to_bf2(a0.x, a0.y);
                        p16[8 + e / 2] = f2_to_bf2(a1.x, a1.y);
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        p16[e] = f2_to_bf2(__uint_as_float(r0[2 * e]) * tv[cb + 2 * e],
                                           __uint_as_float(r0[2 * e + 1]) * tv[cb + 2 * e + 1]);
                        p16[8 + e] = f2_to_bf2(__uint_as_float(r1[2 * e]) * tv[cb + 16 + 2 * e],
                                               __uint_as_float(r1[2 * e + 1]) * tv[cb + 16 + 2 * e + 1]);
                    }
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        r0[e] = __float_as_uint(__uint_as_float(r0[e]) * sg[cb + e]);
                        r1[e] = __float_as_uint(__uint_as_float(r1[e]) * sg[cb + 16 + e]);
                    }
                }
                tmem_st16(tl + T_S16 + cb / 2, p16);
                tmem_st16(tl + T_S + cb, r0);
                tmem_st16(tl + T_S + cb + 16, r1);
            }
            tmem_wait_st();
            tc_fence_before();
            named_bar(NB_EPI, EPI_N);
            if (et == 0) mbar_arrive(s_ready);
            LZ_TRACE(pc, 9);
            // epilogue of the previous chunk (its readout waited for this
            // role's previous iteration only)
            if (pc >= 1 && !epilogue(pc - 1)) { give_up(); break; }
        }
        if (!failed && c_end > c_begin && !epilogue(c_end - c_begin - 1)) give_up();
        // Final state S = Shat F (row i = key dim): Shat^T[j][i] F[i] -> S_out[i][j].
        if (!failed && a.S_out && last_seg) {
            const int nch = c_end - c_begin;
            if (role_wait(warp == W_EPI, lane, NB_EPI_R, EPI_N,
                          [&] { return nch == 0 || bwait(st_done, nch - 1, abort_f); })) {
                tc_fence_after();
                const float *Fv = vec + ((nch - 1) & 1) * NVEC * 128 + 256;
                float *So = a.S_out + (size_t)unit * d * d + j;
#pragma unroll 1
                for (int cc = 0; cc < d; cc += 16) {
                    uint32_t r[16];
                    tmem_ld16(tl + T_S + cc, r);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        if (live)
                            So[(size_t)(cc + e) * d] =
                                nch == 0 ? __uint_as_float(r[e]) : __uint_as_float(r[e]) * Fv[cc + e];
                }
            } else {
                give_up();
            }
        }
    } else if (warp >= W_PREP && warp < W_PREP + 8) {
        // ------------------------------------------------------ gate prep
        // Product form: per element iv = 1 / sigmoid(g) = 1 + 2^{-g log2 e}
        // (= 2^{-lambda}), so the operand scales are running products of iv
        // (no log or exponential per element beyond the one ex2).  Tokens
        // past the end read g = +inf: iv = 1, no decay.
        const int tp = tid - W_PREP * 32;
        const int p = tp & 63, hq = tp >> 6;       // key dims 2p, 2p+1; tokens 16 hq .. 16 hq + 15
        const uint32_t kblk = (p / 32), kbyte = (p % 32) * 4;
        // Gate logits of the chunk being prepared, loaded one chunk ahead
        // (+inf, no decay, past the end and in the padding dims).
        const bool live = 2 * p < d;        // warp-uniform
        const __nv_bfloat16 *gsrc = a.g + (size_t)unit * L * d + 2 * p;
        uint32_t gr[16];
        auto load_g = [&](int c) {
            const int t0 = c * C + 16 * hq;
#pragma unroll
            for (int tt = 0; tt < 16; ++tt)
                gr[tt] = live && t0 + tt < L ? ld_stream_u32(gsrc + (size_t)(t0 + tt) * d) : 0x7F807F80u;
        };
        if (c_begin < c_end) load_g(c_begin);
        float2 Fp = make_float2(1.f, 1.f);         // F of the previous chunk (1: Shat = S at the start)
        for (int c = c_begin; c < c_end; ++c) {
            const int pc = c - c_begin, r = c - c_lo;
            const int s = r % NR, qs = pc % QS, b = pc & 1;
            LZ_TRACE(pc, 0);
            // 1. iv per element and the quarter's product
            float2 iv[16];
            {
                float2 prod = make_float2(1.f, 1.f);
#pragma unroll
                for (int tt = 0; tt < 16; ++tt) {
                    const float2 g2 = bf2_to_f2(gr[tt]);
                    iv[tt] = make_float2(1.f + ex2(g2.x * -LOG2E), 1.f + ex2(g2.y * -LOG2E));
                    prod = mul2(prod, iv[tt]);
                }
                LZ_TRACE(pc, 18);
                if (c + 1 < c_end) load_g(c + 1);
                *reinterpret_cast<float2 *>(tot + hq * 128 + 2 * p) = prod;
            }
            LZ_TRACE(pc, 19);
            named_bar(NB_PREP, PREP_N);
            LZ_TRACE(pc, 20);
            // 2. quarter products: 2^{-r} = T0 T1, 2^{-(b_last - r)} = T2 T3
            float2 T[4];
#pragma unroll
            for (int qq = 0; qq < 4; ++qq) T[qq] = *reinterpret_cast<const float2 *>(tot + qq * 128 + 2 * p);
            const float2 h0 = mul2(T[0], T[1]), h1 = mul2(T[2], T[3]);
            constexpr float SPAN_MAX = 1.2676506e30f;  // 2^SPAN2_MAX
            const bool wide = !(fmaxf(fmaxf(h0.x, h0.y), fmaxf(h1.x, h1.y)) <= SPAN_MAX);
            if (!role_wait(warp == W_PREP, lane, NB_PREP_R, PREP_N, [&] {
                    return bwait(&k_full[s], r / NR, abort_f) && bwait(&q_full[qs], pc / QS, abort_f) &&
                           (pc < 2 || bwait(&op_free[b], (pc >> 1) - 1, abort_f));
                })) { give_up(); break; }
            LZ_TRACE(pc, 21);
            // every prep thread has read tot: the next step may overwrite it
            const bool unsafe = named_bar_or(NB_PREP, PREP_N, wide);
            LZ_TRACE(pc, 1);
            const uint8_t *kraw = sm + SM::KV + s * SLOT + kblk * KB_K;
            const uint8_t *qraw = sm + SM::Q + qs * 2 * KB_T + kblk * KB_T;
            uint8_t *qr_t = sm + SM::OP + b * OPB + kblk * KB_T, *kr_t = qr_t + 2 * KB_T;
            float *vb = vec + b * NVEC * 128;
            if (!unsafe) {
                // Z_t = 2^{r - b_t}: a running product of iv from the start
                // of the thread's half, times 2^r in the first half
                // (2^{r - b_t} = 2^r prod_{0..t} iv there).  KR = k Z,
                // QR = q / Z; every factor lies in [2^-SPAN2_MAX, 2^SPAN2_MAX].
                const float2 er = make_float2(rcp(h0.x), rcp(h0.y));     // 2^r
                float2 R = hq == 0 ? er : hq == 1 ? mul2(er, T[0]) : hq == 2 ? make_float2(1.f, 1.f) : T[2];
                // rolled over blocks of four tokens, iv shifting down by four
                // per block (static register indices): one copy of the body
                // keeps the chunk loop's code small
                if (live)
#pragma unroll 1
                for (int t4 = 0; t4 < 16; t4 += 4) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        R = mul2(R, iv[i]);
                        const uint32_t off = sw128_offset(16 * hq + t4 + i, kbyte);
                        const float2 kv = bf2_to_f2(*reinterpret_cast<const uint32_t *>(kraw + off));
                        const float2 qv = bf2_to_f2(*reinterpret_cast<const uint32_t *>(qraw + off));
                        const float2 kr = mul2(kv, R), qr = mul2(qv, make_float2(rcp(R.x), rcp(R.y)));
                        *reinterpret_cast<uint32_t *>(kr_t + off) = f2_to_bf2(kr.x, kr.y);
                        *reinterpret_cast<uint32_t *>(qr_t + off) = f2_to_bf2(qr.x, qr.y);
                    }
#pragma unroll
                    for (int i = 0; i < 12; ++i) iv[i] = iv[i + 4];
                }
                const float2 F = make_float2(rcp(h1.x), rcp(h1.y));       // 2^{b_last - r}
                const float2 sc = mul2(Fp, er);                              // F_{c-1} 2^r
                if (hq == 0) {
                    *reinterpret_cast<float2 *>(vb + 2 * p) = sc;
                    *reinterpret_cast<float2 *>(vb + 128 + 2 * p) = sc;
                    *reinterpret_cast<float2 *>(vb + 256 + 2 * p) = F;
                }
                Fp = F;
            } else {
                // Exact intra-chunk scores on the CUDA cores, in log space:
                // b_t = sum log2 sigmoid(g) from this chunk's logits (read
                // again: the registers hold the next chunk's by now).
                // Scratch: the other operand buffer holds b (fp32, [64][128])
                // meanwhile; its chunk's products and the previous softmax
                // (which read the A columns) are done.
                if (!role_wait(warp == W_PREP, lane, NB_PREP_R, PREP_N, [&] {
                        return pc == 0 ||
                               (bwait(&op_free[b ^ 1], (pc - 1) >> 1, abort_f) && bwait(sc_free, pc - 1, abort_f));
                    })) { give_up(); break; }
                float *bz = reinterpret_cast<float *>(sm + SM::OP + (b ^ 1) * OPB);
                {
                    // the quarter's prefix sums into the scratch, its total to tot
                    float2 run = make_float2(0.f, 0.f);
                    const int t0 = c * C + 16 * hq;
#pragma unroll 1
                    for (int tt = 0; tt < 16; ++tt) {
                        const uint32_t gv =
                            live && t0 + tt < L ? ld_stream_u32(gsrc + (size_t)(t0 + tt) * d) : 0x7F807F80u;
                        run = add2(run, log2_sigmoid2(bf2_to_f2(gv)));
                        *reinterpret_cast<float2 *>(bz + (16 * hq + tt) * D + 2 * p) = run;
                    }
                    *reinterpret_cast<float2 *>(tot + hq * 128 + 2 * p) = run;
                }
                named_bar(NB_PREP, PREP_N);
                float2 pre = make_float2(0.f, 0.f), blast = make_float2(0.f, 0.f);  // b before the quarter, b_last
#pragma unroll
                for (int qq = 0; qq < 4; ++qq) {
                    const float2 Tq = *reinterpret_cast<const float2 *>(tot + qq * 128 + 2 * p);
                    if (qq < hq) pre = add2(pre, Tq);
                    blast = add2(blast, Tq);
                }
#pragma unroll 1
                for (int tt = 0; tt < 16; ++tt) {
                    float2 *bp = reinterpret_cast<float2 *>(bz + (16 * hq + tt) * D + 2 * p);
                    *bp = add2(*bp, pre);
                }
                named_bar(NB_PREP, PREP_N);
                {
                    const int quarter = warp & 3, li = ((warp - W_PREP) >> 2) * 32 + lane;
                    const int t = 16 * quarter + (li & 15), s0 = 16 * (li >> 4);
                    const uint8_t *qrow = sm + SM::Q + qs * 2 * KB_T;
                    const uint8_t *krow = sm + SM::KV + s * SLOT;
                    float acc[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) acc[e] = 0.f;
                    for (int i = 0; i < d; ++i) {
                        const float qv = __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(
                            qrow + (i / 64) * KB_T + sw128_offset(t, (i % 64) * 2)));
                        const float bt = bz[t * D + i];
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            const int sk = s0 + e;
                            if (sk <= t) {
                                const float kv = __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(
                                    krow + (i / 64) * KB_K + sw128_offset(sk, (i % 64) * 2)));
                                acc[e] += qv * kv * ex2(bt - bz[sk * D + i]);
                            }
                        }
                    }
                    uint32_t rr[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) rr[e] = __float_as_uint(acc[e]);
                    if constexpr (NP == 2) {
                        // A lives in the current chunk's score columns: after the softmax read them
                        if (!role_wait(warp == W_PREP, lane, NB_PREP_R, PREP_N,
                                       [&] { return bwait(sc_read, pc, abort_f); })) { give_up(); break; }
                        tc_fence_after();
                    }
                    tmem_st16_x2<16>(tmem + tlane(quarter) + TM::A + 32 * ((warp - W_PREP) >> 2), rr);
                    tmem_wait_st();
                }
                tc_fence_before();
                named_bar(NB_PREP, PREP_N);
                // QR with r = 0 (exponents <= 0); the key operand is KL, F = 1.
#pragma unroll 1
                for (int tt = 0; tt < 16; ++tt) {
                    const int t = 16 * hq + tt;
                    const uint32_t off = sw128_offset(t, kbyte);
                    const float2 bt = *reinterpret_cast<const float2 *>(bz + t * D + 2 * p);
                    const float2 qv = bf2_to_f2(*reinterpret_cast<const uint32_t *>(qraw + off));
                    const float2 kv = bf2_to_f2(*reinterpret_cast<const uint32_t *>(kraw + off));
                    *reinterpret_cast<uint32_t *>(qr_t + off) = f2_to_bf2(qv.x * ex2(bt.x), qv.y * ex2(bt.y));
                    *reinterpret_cast<uint32_t *>(kr_t + off) =
                        f2_to_bf2(kv.x * ex2(blast.x - bt.x), kv.y * ex2(blast.y - bt.y));
                }
                if (hq == 0) {
                    *reinterpret_cast<float2 *>(vb + 2 * p) = make_float2(Fp.x * ex2(blast.x), Fp.y * ex2(blast.y));
                    *reinterpret_cast<float2 *>(vb + 128 + 2 * p) = Fp;
                    *reinterpret_cast<float2 *>(vb + 256 + 2 * p) = make_float2(1.f, 1.f);
                }
                Fp = make_float2(1.f, 1.f);
            }
            fence_proxy_async_smem();
            named_bar(NB_PREP, PREP_N);
            if (tp == 0) {
                unsafe_f[b] = unsafe ? 1 : 0;
                mbar_arrive(&op_full[b]);
                mbar_arrive(&q_empty[qs]);
            }
            LZ_TRACE(pc, 2);
        }
        // State hand-off: the last min(L, w) keys and values into the ring
        // (token p0 + tau in slot (p0 + tau) % w), pos = L (a continued
        // prompt advanced pos at its start).
        if (!failed && a.S_out && last_seg) {
            const int first = max(0, L - w);
            const __nv_bfloat16 *kp = a.k + (size_t)kvu * L * d, *vp = a.v + (size_t)kvu * L * d;
            __nv_bfloat16 *rk = a.ring_k + (size_t)unit * w * d, *rv = a.ring_v + (size_t)unit * w * d;
            for (int e = tp; e < (L - first) * (d / 8); e += PREP_N) {
                const int tau = first + e / (d / 8), i8 = (e % (d / 8)) * 8;
                const size_t slot = (size_t)((p0 + tau) % w);
                *reinterpret_cast<uint4 *>(rk + slot * d + i8) =
                    *reinterpret_cast<const uint4 *>(kp + (size_t)tau * d + i8);
                *reinterpret_cast<uint4 *>(rv + slot * d + i8) =
                    *reinterpret_cast<const uint4 *>(vp + (size_t)tau * d + i8);
            }
            if (!a.cont && h == 0 && tp == 0) a.pos[unit / a.H] = L;
        }
    } else {
        // ------------------------------------------------------ window softmax
        const int quarter = warp & 3, hs = lane >> 4;
        const int t = 16 * quarter + (lane & 15);
        const uint32_t tl = tmem + tlane(quarter);
        const int st_ = tid - W_SOFT * 32;
        const float alpha = head_alpha(a.alpha_h, a.alpha, h);  // this head's anchor weight
        if constexpr (W64) {
            if (c_lo == c_begin) {
                // no chunk before the first: its score columns read as no
                // key (no product writes them before the first release)
                uint32_t ninf[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) ninf[e] = 0xFF800000u;
#pragma unroll
                for (int cc = 0; cc < 64; cc += 16) tmem_st16(tl + T_SC + cc, ninf);
                tmem_wait_st();
            }
        }
        for (int c = c_begin; c < c_end; ++c) {
            const int pc = c - c_begin;
            const int c0 = c * C, n = min(C, L - c0);
            const bool rowok = t < n;
            const int pbase = c0 - 64 * NP;  // position of band column 0 (the prompt starts at 0)
            // Keys of row t: positions max(-nvalid, tg - w + 1) .. tg, i.e.
            // band columns lo .. hi.
            const int hi = t + 64 * NP, lo = max(-pbase - nvalid, hi - w + 1);
            // (with NP = 2 the A product follows the read of the current
            // chunk's scores, in their columns: waited for below)
            if (!role_wait(warp == W_SOFT, lane, NB_SOFT_R, SOFT_N,
                           [&] { return bwait(sc_full, pc, abort_f) && (NP == 2 || bwait(a_full, pc, abort_f)); })) {
                give_up();
                break;
            }
            LZ_TRACE(pc, 12);
            tc_fence_after();
            // Overlay of the two band chunks (w <= 64): slot s <= t holds
            // current-chunk column s and slot s > t previous-chunk column s.
            // Row t's window keys all sit in distinct slots (exactly the 64
            // slots when w = 64 and the history is complete), so each thread
            // scores 32 slots, not 64.
            bool brk = false, fast = FAST;
            if constexpr (NP == 1 && !FAST) fast = w <= 64;
            if (fast) {
                // Read SC and A first and release their columns at once, so
                // that the next chunk's score products overlap this softmax.
                float x[2][16];
                float mx = -INFINITY;
                uint32_t rm[16], ra2[2][16];
                {
                    uint32_t rp[2][16], rc[2][16];
                    tmem_ld16_x2<16>(tl + T_SC, rp[0]);
                    tmem_ld16_x2<16>(tl + T_SC + 32, rp[1]);
                    tmem_ld16_x2<16>(tl + T_SC + 64, rc[0]);
                    tmem_ld16_x2<16>(tl + T_SC + 96, rc[1]);
                    tmem_ld16(tl + T_SC + 128, rm);
                    tmem_wait_ld();
                    if (W64 || (w == 64 && 64 - c0 - nvalid <= 1)) {
                        // every slot is a key of its row
#pragma unroll
                        for (int jj = 0; jj < 2; ++jj) {
                            const int dj = t - 16 * hs - 32 * jj;  // slot 32 jj + 16 hs + e <= t iff e <= dj
#pragma unroll
                            for (int e = 0; e < 16; ++e) {
                                x[jj][e] = __uint_as_float(e <= dj ? rc[jj][e] : rp[jj][e]);
                                mx = fmaxf(mx, x[jj][e]);
                            }
                        }
                    } else {
                        // slot s is a key iff its band column (64 + s current,
                        // s previous) is at least lo
#pragma unroll
                        for (int jj = 0; jj < 2; ++jj) {
                            const int dj = t - 16 * hs - 32 * jj;
                            const int lc = lo - 64 - 16 * hs - 32 * jj, lp = lo - 16 * hs - 32 * jj;
#pragma unroll
                            for (int e = 0; e < 16; ++e) {
                                const bool cur = e <= dj;
                                const bool key = e >= (cur ? lc : lp);
                                x[jj][e] = key ? __uint_as_float(cur ? rc[jj][e] : rp[jj][e]) : -INFINITY;
                                mx = fmaxf(mx, x[jj][e]);
                            }
                        }
                    }
                }
                tmem_ld16_x2<16>(tl + TM::A, ra2[0]);  // intra-chunk scores A of this thread's slots
                tmem_ld16_x2<16>(tl + TM::A + 32, ra2[1]);
                tmem_wait_ld();
                tc_fence_before();
                named_bar(NB_SOFT, SOFT_N);
                if (st_ == 0) mbar_arrive(sc_free);
                LZ_TRACE(pc, 13);
#pragma unroll
                for (int e = 0; e < META_ROWS; ++e) {
                    if (e >= m) break;
                    if (hs == 0) mx = fmaxf(mx, __uint_as_float(rm[e]));
                }
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                LZ_TRACE(pc, 22);
                const float2 M2 = make_float2(-mx * LOG2E, -mx * LOG2E), L2E = make_float2(LOG2E, LOG2E);
                float2 sum2 = make_float2(0.f, 0.f);
#pragma unroll
                for (int jj = 0; jj < 2; ++jj)
#pragma unroll
                    for (int e = 0; e < 16; e += 2) {
                        const float2 z = fma2(make_float2(x[jj][e], x[jj][e + 1]), L2E, M2);
                        x[jj][e] = ex2(z.x);
                        x[jj][e + 1] = ex2(z.y);
                        sum2 = add2(sum2, make_float2(x[jj][e], x[jj][e + 1]));
                    }
                float sum = sum2.x + sum2.y;
#pragma unroll
                for (int e = 0; e < META_ROWS; ++e) {
                    if (e >= m) break;
                    if (hs == 0) sum += ex2(fmaf(__uint_as_float(rm[e]), LOG2E, M2.x));
                }
                sum += __shfl_xor_sync(0xffffffffu, sum, 16);
                LZ_TRACE(pc, 23);
                const float inv = alpha / sum;
                if (!role_wait(warp == W_SOFT, lane, NB_SOFT_R, SOFT_N,
                               [&] { return pc == 0 || bwait(w_free, pc - 1, abort_f); })) {
                    give_up();
                    break;
                }
                const float2 inv2 = make_float2(rowok ? inv : 0.f, rowok ? inv : 0.f);
                // (a rolled loop: jj picks registers by value, so the code is
                // one copy of the body)
#pragma unroll 1
                for (int jj = 0; jj < 2; ++jj) {
                    const int dj = t - 16 * hs - 32 * jj;
                    uint32_t pp[8], pq[8];
#pragma unroll
                    for (int e = 0; e < 16; e += 2) {
                        const float x0 = jj ? x[1][e] : x[0][e], x1 = jj ? x[1][e + 1] : x[0][e + 1];
                        const uint32_t a0 = jj ? ra2[1][e] : ra2[0][e], a1 = jj ? ra2[1][e + 1] : ra2[0][e + 1];
                        const float2 v = mul2(make_float2(x0, x1), inv2);
                        const float2 av = make_float2(rowok ? __uint_as_float(a0) : 0.f,
                                                      rowok ? __uint_as_float(a1) : 0.f);
                        const float2 vc = add2(v, av);
                        const bool c0_ = e <= dj, c1_ = e + 1 <= dj;
                        pp[e / 2] = f2_to_bf2(c0_ ? 0.f : v.x, c1_ ? 0.f : v.y);
                        pq[e / 2] = f2_to_bf2(c0_ ? vc.x : 0.f, c1_ ? vc.y : 0.f);
                    }
                    const int col = 32 * jj + 16 * hs;
                    *reinterpret_cast<uint4 *>(sm + SM::W + sw128_offset(t, col * 2)) = make_uint4(pp[0], pp[1], pp[2], pp[3]);
                    *reinterpret_cast<uint4 *>(sm + SM::W + sw128_offset(t, col * 2 + 16)) = make_uint4(pp[4], pp[5], pp[6], pp[7]);
                    *reinterpret_cast<uint4 *>(sm + SM::W + KB_T + sw128_offset(t, col * 2)) = make_uint4(pq[0], pq[1], pq[2], pq[3]);
                    *reinterpret_cast<uint4 *>(sm + SM::W + KB_T + sw128_offset(t, col * 2 + 16)) = make_uint4(pq[4], pq[5], pq[6], pq[7]);
                }
            } else if constexpr (!FAST) {
                // Every band column scored separately (w = 65, a window of
                // one token, or two earlier band chunks), in three passes over
                // tensor memory -- max, sum, weights -- so that one 16-column
                // group is held at a time.
                const int d0 = 16 * hs - lo;
                const uint32_t span = (uint32_t)(hi - lo);
                uint32_t rm[16];
                tmem_ld16(tl + T_SC + 64 * NB, rm);
                float mx = -INFINITY;
#pragma unroll 1
                for (int jj = 0; jj < 2 * NB; ++jj) {
                    uint32_t r[16];
                    tmem_ld16_x2<16>(tl + T_SC + 32 * jj, r);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        if ((uint32_t)(d0 + 32 * jj + e) <= span) mx = fmaxf(mx, __uint_as_float(r[e]));
                }
#pragma unroll
                for (int e = 0; e < META_ROWS; ++e) {
                    if (e >= m) break;
                    if (hs == 0) mx = fmaxf(mx, __uint_as_float(rm[e]));
                }
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                LZ_TRACE(pc, 22);
                const float M2 = mx * LOG2E;
                float sum = 0.f;
#pragma unroll 1
                for (int jj = 0; jj < 2 * NB; ++jj) {
                    uint32_t r[16];
                    tmem_ld16_x2<16>(tl + T_SC + 32 * jj, r);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        if ((uint32_t)(d0 + 32 * jj + e) <= span) sum += ex2(fmaf(__uint_as_float(r[e]), LOG2E, -M2));
                }
#pragma unroll
                for (int e = 0; e < META_ROWS; ++e) {
                    if (e >= m) break;
                    if (hs == 0) sum += ex2(fmaf(__uint_as_float(rm[e]), LOG2E, -M2));
                }
                sum += __shfl_xor_sync(0xffffffffu, sum, 16);
                LZ_TRACE(pc, 23);
                const float inv = alpha / sum;
                if (!role_wait(warp == W_SOFT, lane, NB_SOFT_R, SOFT_N,
                               [&] { return pc == 0 || bwait(w_free, pc - 1, abort_f); })) {
                    give_up();
                    brk = true;
                }
                if (!brk) {
                    // W = alpha P / Z, plus A (s <= t) in the current chunk's columns
                    constexpr int JW = NP == 2 ? 2 * NP : 2 * NB;  // groups done here
#pragma unroll 1
                    for (int jj = 0; jj < JW; ++jj) {
                        const bool cur = jj >= 2 * NP;
                        uint32_t r[16], ra[16];
                        tmem_ld16_x2<16>(tl + T_SC + 32 * jj, r);
                        tmem_ld16_x2<16>(tl + TM::A + 32 * (cur ? jj - 2 * NP : 0), ra);
                        tmem_wait_ld();
                        const int col0 = 32 * jj + 16 * hs;
                        uint32_t pk[8];
#pragma unroll
                        for (int e = 0; e < 16; e += 2) {
                            float wv[2];
#pragma unroll
                            for (int u = 0; u < 2; ++u) {
                                const bool key = (uint32_t)(d0 + 32 * jj + e + u) <= span;
                                float v = key ? ex2(fmaf(__uint_as_float(r[e + u]), LOG2E, -M2)) * inv : 0.f;
                                if (cur && col0 + e + u - 64 * NP <= t) v += __uint_as_float(ra[e + u]);
                                wv[u] = rowok ? v : 0.f;
                            }
                            pk[e / 2] = f2_to_bf2(wv[0], wv[1]);
                        }
                        const uint32_t blk = (col0 / 64) * KB_T, byte = (col0 % 64) * 2;
                        *reinterpret_cast<uint4 *>(sm + SM::W + blk + sw128_offset(t, byte)) =
                            make_uint4(pk[0], pk[1], pk[2], pk[3]);
                        *reinterpret_cast<uint4 *>(sm + SM::W + blk + sw128_offset(t, byte + 16)) =
                            make_uint4(pk[4], pk[5], pk[6], pk[7]);
                    }
                    if constexpr (NP == 2) {
                        // The current chunk: its weights to registers, its
                        // columns released to the A product (A is accumulated
                        // in them), then A added.
                        float pv[2][16];
#pragma unroll
                        for (int jx = 0; jx < 2; ++jx) {
                            const int jj = 2 * NP + jx;
                            uint32_t r[16];
                            tmem_ld16_x2<16>(tl + T_SC + 32 * jj, r);
                            tmem_wait_ld();
#pragma unroll
                            for (int e = 0; e < 16; ++e)
                                pv[jx][e] = (uint32_t)(d0 + 32 * jj + e) <= span
                                                ? ex2(fmaf(__uint_as_float(r[e]), LOG2E, -M2)) * inv
                                                : 0.f;
                        }
                        tc_fence_before();
                        named_bar(NB_SOFT, SOFT_N);
                        if (st_ == 0) mbar_arrive(sc_read);
                        if (!role_wait(warp == W_SOFT, lane, NB_SOFT_R, SOFT_N,
                                       [&] { return bwait(a_full, pc, abort_f); })) {
                            give_up();
                            brk = true;
                        }
                        if (!brk) {
                            tc_fence_after();
                            uint32_t ra[2][16];
                            tmem_ld16_x2<16>(tl + TM::A, ra[0]);
                            tmem_ld16_x2<16>(tl + TM::A + 32, ra[1]);
                            tmem_wait_ld();
#pragma unroll
                            for (int jx = 0; jx < 2; ++jx) {
                                const int col0 = 32 * (2 * NP + jx) + 16 * hs;
                                uint32_t pk[8];
#pragma unroll
                                for (int e = 0; e < 16; e += 2) {
                                    float wv[2];
#pragma unroll
                                    for (int u = 0; u < 2; ++u) {
                                        float v = pv[jx][e + u];
                                        if (col0 + e + u - 64 * NP <= t) v += __uint_as_float(ra[jx][e + u]);
                                        wv[u] = rowok ? v : 0.f;
                                    }
                                    pk[e / 2] = f2_to_bf2(wv[0], wv[1]);
                                }
                                const uint32_t blk = (col0 / 64) * KB_T, byte = (col0 % 64) * 2;
                                *reinterpret_cast<uint4 *>(sm + SM::W + blk + sw128_offset(t, byte)) =
                                    make_uint4(pk[0], pk[1], pk[2], pk[3]);
                                *reinterpret_cast<uint4 *>(sm + SM::W + blk + sw128_offset(t, byte + 16)) =
                                    make_uint4(pk[4], pk[5], pk[6], pk[7]);
                            }
                        }
                    }
                    if (!brk) {
                        // SC and A are read: the next chunk's scores may overwrite them
                        tc_fence_before();
                        named_bar(NB_SOFT, SOFT_N);
                        if (st_ == 0) mbar_arrive(sc_free);
                        LZ_TRACE(pc, 13);
                    }
                }
            }
            if (brk) break;
            fence_proxy_async_smem();
            named_bar(NB_SOFT, SOFT_N);
            if (st_ == 0) mbar_arrive(w_full);
            LZ_TRACE(pc, 14);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == W_MMA) tmem_dealloc(tmem, 512);
}

}  // namespace ws
}  // namespace lizard
