// lizard_attn.cu -- C ABI of the Lizard hybrid attention operator.
//
// Host-side validation and launch of the kernels in decode.cuh,
// prefill_ws.cuh (bf16, d = 128 with any window, d = 64 with w <= 65:
// warp-specialised tensor cores, with the segment pre-pass of
// prefill_state.cuh for d = 128), prefill_simt.cuh (fp32, and bf16 d = 64
// with w > 65: CUDA cores, exact fp32), prefill_cont.cuh (start position of a continued prompt),
// backward_simt.cuh / backward_tc.cuh (gradients), gate_proj.cuh (the gate
// projection) and the state initialiser below.  Declarations and the contract of every entry point are
// in include/lizard_attn.h.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "../../include/lizard_attn.h"
#include "common.cuh"
#include "decode.cuh"
#include "prefill_simt.cuh"
#include "prefill_ws.cuh"
#include "prefill_state.cuh"
#include "prefill_cont.cuh"
#include "backward_simt.cuh"
#include "backward_tc.cuh"
#include "gate_proj.cuh"

namespace lizard {

__global__ void state_init_kernel(float *S, size_t nS, uint4 *ring_k, uint4 *ring_v, size_t nring16,
                                  int64_t *pos, int B)
{
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    const size_t i0 = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
    for (size_t i = i0; i < nS / 4; i += stride) reinterpret_cast<float4 *>(S)[i] = z4;
    const uint4 zu = make_uint4(0, 0, 0, 0);
    for (size_t i = i0; i < nring16; i += stride) {
        ring_k[i] = zu;
        ring_v[i] = zu;
    }
    for (size_t i = i0; i < (size_t)B; i += stride) pos[i] = 0;
}

static bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
static bool aligned8(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 7u) == 0; }

// Stream-ordered scratch from a memory pool this library owns, one per
// device.  Its release threshold is unlimited: memory a call frees stays
// reserved for the library's next calls, so a steady stream of calls maps
// no new memory (the device's default pool would hand freed memory back at
// every synchronisation), until lizard_scratch_trim returns it.  The
// caller's own allocations are untouched.
static std::mutex g_pool_mu;
static constexpr int MAX_POOL_DEV = 64;
static cudaMemPool_t g_pools[MAX_POOL_DEV] = {};

// The library's pool on device `dev`, created on first use when `create`.
static cudaError_t scratch_pool(int dev, bool create, cudaMemPool_t *out)
{
    *out = nullptr;
    if (dev < 0 || dev >= MAX_POOL_DEV) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_pool_mu);
    if (!g_pools[dev] && create) {
        cudaMemPoolProps props = {};
        props.allocType = cudaMemAllocationTypePinned;
        props.handleTypes = cudaMemHandleTypeNone;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        cudaMemPool_t np = nullptr;
        cudaError_t e = cudaMemPoolCreate(&np, &props);
        if (e != cudaSuccess) return e;
        uint64_t keep = UINT64_MAX;
        e = cudaMemPoolSetAttribute(np, cudaMemPoolAttrReleaseThreshold, &keep);
        if (e != cudaSuccess) {
            cudaMemPoolDestroy(np);
            return e;
        }
        g_pools[dev] = np;
    }
    *out = g_pools[dev];
    return cudaSuccess;
}

static cudaError_t scratch_alloc(void **p, size_t bytes, cudaStream_t s)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    cudaMemPool_t pool;
    e = scratch_pool(dev, true, &pool);
    if (e != cudaSuccess) return e;
    return cudaMallocFromPoolAsync(p, bytes, pool, s);
}
static size_t esize(lizard_dtype dt) { return dt == LIZARD_F32 ? 4 : 2; }
static bool dtype_ok(lizard_dtype dt) { return dt == LIZARD_F32 || dt == LIZARD_BF16; }

static lizard_status check_state(const lizard_state *st)
{
    if (!st) return LIZARD_ERR_INVALID_ARG;
    if (!dtype_ok(st->dtype)) return LIZARD_ERR_INVALID_ARG;
    if (st->B < 0 || st->H < 1 || st->dk < 1 || st->dv < 1 || st->w < 1) return LIZARD_ERR_INVALID_ARG;
    if (!st->S || !st->ring_k || !st->ring_v || !st->pos) return LIZARD_ERR_INVALID_ARG;
    // pos is one int64 per sequence: 8-byte alignment, so that the state of
    // a slice of the batch (pos + b0) is a valid state too
    if (!aligned16(st->S) || !aligned16(st->ring_k) || !aligned16(st->ring_v) || !aligned8(st->pos))
        return LIZARD_ERR_INVALID_ARG;
    if (st->dk != st->dv || (st->dk != 64 && st->dk != 128 && st->dk != 256)) return LIZARD_ERR_UNSUPPORTED;
    if (st->w > LIZARD_MAX_WINDOW) return LIZARD_ERR_UNSUPPORTED;
    return LIZARD_OK;
}

static lizard_status launch_status()
{
    return cudaGetLastError() == cudaSuccess ? LIZARD_OK : LIZARD_ERR_CUDA;
}

template <typename T, int D>
static lizard_status launch_prefill(const PrefillArgs &pa, cudaStream_t s)
{
    const size_t smem = prefill_simt_smem_bytes<D>(pa.w, pa.m);
    auto kern = prefill_simt_kernel<T, D>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return LIZARD_ERR_CUDA;
    constexpr int NSL = SimtShape<D>::NSL;
    kern<<<pa.B * pa.H * NSL, SIMT_THREADS, smem, s>>>(pa);
    if constexpr (NSL > 1) {
        if (pa.S_out) {
            if (launch_status() != LIZARD_OK) return LIZARD_ERR_CUDA;
            ring_handoff_kernel<T, D><<<pa.B * pa.H, SIMT_THREADS, 0, s>>>(pa);
        }
    }
    return launch_status();
}

typedef CUresult (*encode_tiled_fn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                    const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                    CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, looked up once (a function-local static
// is initialised exactly once even when host threads race to first use).
static encode_tiled_fn lookup_tensor_map_encoder()
{
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
        return reinterpret_cast<encode_tiled_fn>(p);
    return nullptr;
}

static encode_tiled_fn tensor_map_encoder()
{
    static const encode_tiled_fn fn = lookup_tensor_map_encoder();
    return fn;
}

// [units][L][d] bf16 (d = 128 or 64) viewed as a 3-D tensor; 64 x 64 boxes,
// 128B swizzle, rows past L read as zero.
static bool make_token_map(CUtensorMap *map, const void *base, int units, int L, int d = 128)
{
    encode_tiled_fn enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)L, (cuuint64_t)units};
    cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)L * d * 2};
    cuuint32_t box[3] = {64, 64, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int NP, int DH>
static lizard_status launch_prefill_ws_np(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                                          const ws::WsArgs &wa, int ctas, cudaStream_t s)
{
    // w <= 64 with one earlier band chunk: the instance with only the
    // one-overlay softmax compiled in; w = 64 from the empty state: the one
    // without the masked selection either
    auto kern = ws::prefill_ws_kernel<NP, DH, false>;
    if constexpr (NP == 1) {
        if (wa.w == 64 && !wa.cont)
            kern = ws::prefill_ws_kernel<NP, DH, true, true>;
        else if (wa.w <= 64)
            kern = ws::prefill_ws_kernel<NP, DH, true>;
    }
    constexpr uint32_t smem = ws::Smem<NP>::BYTES;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return LIZARD_ERR_CUDA;
    kern<<<ctas, ws::THREADS, smem, s>>>(tq, tk, tv, wa);
    return launch_status();
}

static int sm_count()
{
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 1;
    return n > 0 ? n : 1;
}

// Sequence segments per (batch, head) unit: enough CTAs to cover the SMs
// when there are few units, each segment at least 8 chunks long.
static int prefill_segments(int units, int nchunks)
{
    const int p = sm_count() / (units > 0 ? units : 1);
    const int cap = nchunks / 8;
    return p < 1 || cap < 1 ? 1 : (p < cap ? p : cap);
}

// Scratch of a segmented prefill, in order: the segments' start states
// [units][nseg-1][D][D] (what the prefill reads); with sub-blocks (nsub > 1)
// the sub-blocks' end states [units][(nseg-1) nsub][D][D] (with nsub = 1
// they share the start states' space: the scan writes each over what it
// has just read); the decays [units][(nseg-1) nsub][D]; for a continued
// prompt copies of its start state and window history.  All fp32 but the
// history (bf16); every offset a multiple of 16 bytes.
struct SegLayout {
    size_t sub_off, lam_off, cont_off, total;
};
static SegLayout segment_layout(int units, int nseg, int nsub, bool cont)
{
    const size_t DD = (size_t)ws::D * ws::D * sizeof(float), nsp = (size_t)units * (nseg - 1);
    SegLayout l;
    l.sub_off = nsub > 1 ? nsp * DD : 0;
    l.lam_off = nsp * DD + (nsub > 1 ? nsp * nsub * DD : 0);
    l.cont_off = l.lam_off + nsp * nsub * ws::D * sizeof(float);
    l.total = l.cont_off + (cont ? (size_t)units * (DD + 2 * ws::C * ws::D * sizeof(__nv_bfloat16)) : 0);
    return l;
}

// Sub-blocks per segment in the pre-pass: the count (1..8) whose CTAs, in
// whole waves over the SMs (one pre-pass CTA per SM), walk the fewest chunks
// one after another; ties go to fewer sub-blocks.
static int segment_subblocks(int units, int nseg, int seg_chunks)
{
    const long long sms = sm_count(), ctas = (long long)units * (nseg - 1);
    int best = 1;
    long long best_cost = -1;
    for (int nsub = 1; nsub <= 8 && nsub <= seg_chunks; ++nsub) {
        const long long cost = ((ctas * nsub + sms - 1) / sms) * ((seg_chunks + nsub - 1) / nsub);
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best = nsub;
        }
    }
    return best;
}

// The segment pre-pass: end state and total decay of every segment but the
// last, then the start state of every segment (written over the end states).
// For a continued prompt `sc` names its start state and the copies the
// first segment reads.
static lizard_status launch_segment_states(const CUtensorMap &tk, const CUtensorMap &tv, const CUtensorMap &tg,
                                           float *scratch, const SegLayout &lay, int nsub, int units, int L,
                                           int seg_chunks, int nseg, const seg::ScanCont &sc, int H, int group,
                                           cudaStream_t s)
{
    uint8_t *base = reinterpret_cast<uint8_t *>(scratch);
    seg::SegArgs sa{reinterpret_cast<float *>(base + lay.sub_off), reinterpret_cast<float *>(base + lay.lam_off),
                    L, seg_chunks, nseg, H, group, nsub, (seg_chunks + nsub - 1) / nsub};
    if (cudaFuncSetAttribute(seg::segment_state_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)seg::SMEM_BYTES) != cudaSuccess)
        return LIZARD_ERR_CUDA;
    seg::segment_state_kernel<<<units * (nseg - 1) * nsub, seg::THREADS, seg::SMEM_BYTES, s>>>(tk, tv, tg, sa);
    if (cudaGetLastError() != cudaSuccess) return LIZARD_ERR_CUDA;
    seg::segment_scan_kernel<<<dim3(ws::D * ws::D / 256, units), 256, 0, s>>>(sa.dS, sa.lam, scratch, units, nseg,
                                                                              nsub, sc);
    return launch_status();
}

// Warp-specialised tensor-core prefill (bf16; d = 128, any window; d = 64,
// w <= 65).  With few (batch, head) units and a long prompt the sequence
// (d = 128) is split into segments that run side by side, after a pre-pass
// that computes every segment's start state; `scratch` (nullable) holds
// those states, else they live in stream-ordered scratch from the library's
// pool (freed on `s`).  d = 64 runs one CTA per unit on the same tiles,
// zero-padded.
static lizard_status launch_prefill_ws(const PrefillArgs &pa, cudaStream_t s, float *scratch = nullptr,
                                       size_t scratch_bytes = 0, int force_segments = 0, int d = 128)
{
    const int units = pa.B * pa.H;
    const int nchunks = (pa.L + ws::C - 1) / ws::C;
    // d = 64, and a continued prompt with a two-chunk band: one CTA per unit
    // (the segment copies hold one chunk of window history)
    const bool one_seg = d != ws::D || (pa.cont && pa.w > 65);
    int nseg = one_seg ? 1 : force_segments > 0 ? force_segments : prefill_segments(units, nchunks);
    if (nseg > nchunks) nseg = nchunks;
    const int seg_chunks = (nchunks + nseg - 1) / (nseg > 0 ? nseg : 1);
    nseg = seg_chunks > 0 ? (nchunks + seg_chunks - 1) / seg_chunks : 1;  // no empty segment
    if (nseg < 1) nseg = 1;
    const int kv_units = pa.B * (pa.H / pa.group);
    CUtensorMap tq, tk, tv, tg;
    if (!make_token_map(&tq, pa.q, units, pa.L, d) || !make_token_map(&tk, pa.k, kv_units, pa.L, d) ||
        !make_token_map(&tv, pa.v, kv_units, pa.L, d) || !make_token_map(&tg, pa.g, units, pa.L, d))
        return LIZARD_ERR_CUDA;
    float *seg_states = nullptr;
    int nsub = 1;
    SegLayout lay{};
    bool owned = false;
    if (nseg > 1) {
        nsub = segment_subblocks(units, nseg, seg_chunks);
        lay = segment_layout(units, nseg, nsub, pa.cont != 0);
        if (scratch && scratch_bytes < lay.total) {  // the allocation-free call's fixed array: whole segments
            nsub = 1;
            lay = segment_layout(units, nseg, nsub, pa.cont != 0);
        }
        const size_t need = lay.total;
        if (scratch) {
            if (scratch_bytes < need) return LIZARD_ERR_UNSUPPORTED;
            seg_states = scratch;
        } else if (scratch_alloc(reinterpret_cast<void **>(&seg_states), need, s) == cudaSuccess) {
            owned = true;
        } else {
            cudaGetLastError();
            nseg = 1;  // no scratch to be had: one CTA per unit walks the whole prompt
        }
    }
    lizard_status rc = LIZARD_OK;
    // Start state and window history of the first segment: read in place
    // when one CTA walks the whole prompt (it reads them before it writes the
    // state), else copies that the scan makes.
    const float *seg0_state = pa.S0;
    const __nv_bfloat16 *hist = nullptr;
    if (nseg > 1) {
        seg::ScanCont sc{};
        if (pa.cont) {
            float *copy = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(seg_states) + lay.cont_off);
            __nv_bfloat16 *hcopy = reinterpret_cast<__nv_bfloat16 *>(copy + (size_t)units * ws::D * ws::D);
            sc = seg::ScanCont{pa.S0, copy, static_cast<const __nv_bfloat16 *>(pa.ring_k),
                               static_cast<const __nv_bfloat16 *>(pa.ring_v), pa.pos, hcopy, pa.H, pa.w};
            seg0_state = copy;
            hist = hcopy;
        }
        rc = launch_segment_states(tk, tv, tg, seg_states, lay, nsub, units, pa.L, seg_chunks, nseg, sc, pa.H,
                                   pa.group, s);
    }
    ws::WsArgs wa{static_cast<const __nv_bfloat16 *>(pa.g), static_cast<const __nv_bfloat16 *>(pa.mu),
                  static_cast<const __nv_bfloat16 *>(pa.k), static_cast<const __nv_bfloat16 *>(pa.v),
                  static_cast<__nv_bfloat16 *>(pa.y), pa.S_out, static_cast<__nv_bfloat16 *>(pa.ring_k),
                  static_cast<__nv_bfloat16 *>(pa.ring_v), pa.pos, pa.alpha, pa.H, pa.L, pa.w, pa.m,
                  nseg > 1 ? seg_states : nullptr, nseg > 1 ? seg_chunks : nchunks, nseg,
                  pa.cont, seg0_state, hist, pa.alpha_h, pa.group};
    if (rc == LIZARD_OK)
        rc = d == ws::D ? (pa.w == 1   ? launch_prefill_ws_np<0, ws::D>(tq, tk, tv, wa, units * nseg, s)
                           : pa.w <= 65 ? launch_prefill_ws_np<1, ws::D>(tq, tk, tv, wa, units * nseg, s)
                                        : launch_prefill_ws_np<2, ws::D>(tq, tk, tv, wa, units * nseg, s))
                        : (pa.w == 1   ? launch_prefill_ws_np<0, 64>(tq, tk, tv, wa, units * nseg, s)
                           : pa.w <= 65 ? launch_prefill_ws_np<1, 64>(tq, tk, tv, wa, units * nseg, s)
                                        : launch_prefill_ws_np<2, 64>(tq, tk, tv, wa, units * nseg, s));
    if (owned && cudaFreeAsync(seg_states, s) != cudaSuccess && rc == LIZARD_OK) rc = LIZARD_ERR_CUDA;
    return rc;
}

// Failure-detection testing: LIZARD_DEBUG_DECODE_FIRST_WAIT_POLLS=n (read
// once per process) makes every decode step give up its first wait after n
// polls and report LIZARD_ERR_TIMEOUT; unset, the normal limit applies.
static int decode_first_wait_polls()
{
    static const int polls = [] {
        const char *e = std::getenv("LIZARD_DEBUG_DECODE_FIRST_WAIT_POLLS");
        return e && *e ? std::atoi(e) : -1;
    }();
    return polls;
}

template <typename T, int D>
static lizard_status launch_decode(DecodeArgs da, cudaStream_t s)
{
    da.first_wait_polls = decode_first_wait_polls();
    const DecodePlan plan = decode_plan<D>((int)sizeof(T), da.w, da.m);
    if (plan.total > DECODE_SMEM_MAX) return LIZARD_ERR_UNSUPPORTED;
    auto kern = decode_step_kernel<T, D>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)plan.total) != cudaSuccess)
        return LIZARD_ERR_CUDA;
    // Programmatic dependent launch: this step's CTAs may start while the
    // previous kernel on the stream drains; the kernel waits for it
    // (griddepcontrol.wait) before touching any data.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(da.B * da.H * decode_split<D>()));
    cfg.blockDim = dim3(DECODE_THREADS);
    cfg.dynamicSmemBytes = plan.total;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kern, da) != cudaSuccess) return LIZARD_ERR_CUDA;
    return launch_status();
}

// Grouped key/value heads: sum the per-query-head dk, dv (ba.dk, ba.dv) of
// each group into the key/value heads' outputs.
template <typename T, int D>
static lizard_status launch_gqa_reduce(const BackwardArgs &ba, void *dk_out, void *dv_out, cudaStream_t s)
{
    const long long LD = (long long)ba.L * D;
    const long long n = (long long)ba.B * (ba.H / ba.group) * LD;
    const int blocks = (int)(n / 256 + 1 < 148LL * 32 ? n / 256 + 1 : 148LL * 32);
    gqa_reduce_kernel<T><<<blocks, 256, 0, s>>>(static_cast<const T *>(ba.dk), static_cast<T *>(dk_out), ba.B, ba.H,
                                                 ba.group, LD);
    gqa_reduce_kernel<T><<<blocks, 256, 0, s>>>(static_cast<const T *>(ba.dv), static_cast<T *>(dv_out), ba.B, ba.H,
                                                 ba.group, LD);
    return launch_status();
}

// Gradients: the two-sweep kernel over every unit, then the reduction of the
// per-unit d mu and d alpha parts.  Scratch from the library's pool.
template <typename T, int D>
static lizard_status launch_backward(BackwardArgs ba, float *dmu, float *dalpha, cudaStream_t s)
{
    const size_t units = (size_t)ba.B * ba.H;
    const size_t xq_bytes = units * ba.L * D * sizeof(float);
    const size_t row_bytes = units * ba.L * sizeof(float);
    const size_t dmu_bytes = units * ba.m * D * sizeof(float);
    // grouped key/value heads: dk, dv per query head first, summed after
    const size_t gqa_bytes = ba.group > 1 ? 2 * ((units * ba.L * D * sizeof(T) + 255) & ~(size_t)255) : 0;
    const size_t bytes = gqa_bytes + xq_bytes + 2 * row_bytes + dmu_bytes + units * sizeof(float);
    uint8_t *scratch = nullptr;
    if (scratch_alloc(reinterpret_cast<void **>(&scratch), bytes, s) != cudaSuccess) {
        cudaGetLastError();
        return LIZARD_ERR_CUDA;
    }
    void *dk_out = ba.dk, *dv_out = ba.dv;
    if (gqa_bytes) {
        ba.dk = scratch;
        ba.dv = scratch + gqa_bytes / 2;
    }
    uint8_t *sc = scratch + gqa_bytes;
    ba.xq = reinterpret_cast<float *>(sc);
    ba.lse = reinterpret_cast<float *>(sc + xq_bytes);
    ba.drow = reinterpret_cast<float *>(sc + xq_bytes + row_bytes);
    ba.dmu_part = reinterpret_cast<float *>(sc + xq_bytes + 2 * row_bytes);
    ba.dalpha_part = reinterpret_cast<float *>(sc + xq_bytes + 2 * row_bytes + dmu_bytes);
    lizard_status rc = LIZARD_OK;
    const size_t smem = backward_simt_smem_bytes<D>(ba.w, ba.m);
    auto kern = backward_simt_kernel<T, D>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) {
        rc = LIZARD_ERR_CUDA;
    } else {
        kern<<<(unsigned)units, BW_THREADS, smem, s>>>(ba);
        rc = launch_status();
    }
    if (rc == LIZARD_OK) {
        const int mD = ba.m * D, n = ba.H * mD;
        backward_reduce_kernel<<<n > 0 ? (n + 255) / 256 : 1, 256, 0, s>>>(ba.dmu_part, ba.dalpha_part, ba.B, ba.H,
                                                                           mD, dmu, dalpha, ba.alpha_h != nullptr);
        rc = launch_status();
    }
    if (rc == LIZARD_OK && gqa_bytes) rc = launch_gqa_reduce<T, D>(ba, dk_out, dv_out, s);
    if (cudaFreeAsync(scratch, s) != cudaSuccess && rc == LIZARD_OK) rc = LIZARD_ERR_CUDA;
    return rc;
}

// Gradients on the tensor cores (bf16, d = 128, w <= 65): the chunk states
// and state gradients, then the query-side and key-side kernels over every
// (unit, chunk).  d mu and d alpha are accumulated, so they start at zero.
// DH: the head dim (128, or 64 on the same zero-padded tiles); the scratch
// keeps the 128-wide layout.
template <int DH>
static lizard_status launch_backward_tc(const BackwardArgs &ba, float *dmu, float *dalpha, cudaStream_t s)
{
    const int units = ba.B * ba.H, L = ba.L, nch = (L + bwdtc::C - 1) / bwdtc::C;
    const int kv_units = ba.B * (ba.H / ba.group);
    const size_t D = bwdtc::D;
    const size_t st_bytes = (size_t)units * nch * D * D * sizeof(__nv_bfloat16);
    const size_t xq_bytes = (size_t)units * L * D * sizeof(float);
    const size_t row_bytes = ((size_t)units * L * sizeof(float) + 255) & ~(size_t)255;
    // grouped key/value heads: dk, dv per query head first, summed after
    const size_t gqa_bytes = ba.group > 1 ? 2 * (size_t)units * L * DH * sizeof(__nv_bfloat16) : 0;
    uint8_t *scratch = nullptr;
    if (scratch_alloc(reinterpret_cast<void **>(&scratch), 2 * st_bytes + xq_bytes + 2 * row_bytes + gqa_bytes, s) !=
        cudaSuccess) {
        cudaGetLastError();
        return LIZARD_ERR_CUDA;
    }
    BackwardArgs bg = ba;
    if (gqa_bytes) {
        bg.dk = scratch + 2 * st_bytes + xq_bytes + 2 * row_bytes;
        bg.dv = static_cast<uint8_t *>(bg.dk) + gqa_bytes / 2;
    }
    __nv_bfloat16 *Sb = reinterpret_cast<__nv_bfloat16 *>(scratch);
    __nv_bfloat16 *Ha = reinterpret_cast<__nv_bfloat16 *>(scratch + st_bytes);
    float *xq = reinterpret_cast<float *>(scratch + 2 * st_bytes);
    float *lse2 = reinterpret_cast<float *>(scratch + 2 * st_bytes + xq_bytes);
    float *drow = reinterpret_cast<float *>(scratch + 2 * st_bytes + xq_bytes + row_bytes);
    lizard_status rc = LIZARD_OK;
    CUtensorMap tq, tk, tv, tg, tdy, tS, tH;
    if (!make_token_map(&tq, ba.q, units, L, DH) || !make_token_map(&tk, ba.k, kv_units, L, DH) ||
        !make_token_map(&tv, ba.v, kv_units, L, DH) || !make_token_map(&tg, ba.g, units, L, DH) ||
        !make_token_map(&tdy, ba.dy, units, L, DH) || !make_token_map(&tS, Sb, units * nch, (int)D) ||
        !make_token_map(&tH, Ha, units * nch, (int)D))
        rc = LIZARD_ERR_CUDA;
    if (rc == LIZARD_OK && cudaMemsetAsync(dalpha, 0, sizeof(float) * (ba.alpha_h ? ba.H : 1), s) != cudaSuccess)
        rc = LIZARD_ERR_CUDA;
    if (rc == LIZARD_OK && dmu && cudaMemsetAsync(dmu, 0, sizeof(float) * ba.H * ba.m * DH, s) != cudaSuccess)
        rc = LIZARD_ERR_CUDA;
    if (rc == LIZARD_OK) {
        bwdtc::StatesArgs sa{Sb, Ha, static_cast<const __nv_bfloat16 *>(ba.g), L, nch, ba.H, ba.group};
        if (cudaFuncSetAttribute(bwdtc::chunk_states_kernel<DH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)bwdtc::ST_SMEM) != cudaSuccess)
            rc = LIZARD_ERR_CUDA;
        else {
            bwdtc::chunk_states_kernel<DH><<<dim3(units, 2), bwdtc::THREADS, bwdtc::ST_SMEM, s>>>(tg, tk, tv, tq, tdy, sa);
            rc = launch_status();
        }
    }
    if (rc == LIZARD_OK) {
        bwdtc::QueryArgs qa{static_cast<const __nv_bfloat16 *>(ba.mu), static_cast<const __nv_bfloat16 *>(ba.k),
                            static_cast<__nv_bfloat16 *>(ba.dq), xq, lse2, drow, dmu, dalpha, ba.alpha, ba.H, L,
                            ba.w, ba.m, nch, ba.alpha_h, ba.group};
        if (cudaFuncSetAttribute(bwdtc::bwd_query_kernel<DH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)bwdtc::QO_SMEM) != cudaSuccess)
            rc = LIZARD_ERR_CUDA;
        else {
            bwdtc::bwd_query_kernel<DH><<<units * nch, bwdtc::THREADS, bwdtc::QO_SMEM, s>>>(tq, tk, tv, tg, tdy, tS, qa);
            rc = launch_status();
        }
    }
    if (rc == LIZARD_OK) {
        bwdtc::KeyArgs ka{Sb, xq, lse2, drow, static_cast<__nv_bfloat16 *>(bg.dk), static_cast<__nv_bfloat16 *>(bg.dv),
                          static_cast<__nv_bfloat16 *>(ba.dg), ba.alpha, L, ba.w, nch, ba.alpha_h, ba.H, ba.group};
        if (cudaFuncSetAttribute(bwdtc::bwd_key_kernel<DH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)bwdtc::KO_SMEM) != cudaSuccess)
            rc = LIZARD_ERR_CUDA;
        else {
            bwdtc::bwd_key_kernel<DH><<<units * nch, bwdtc::THREADS, bwdtc::KO_SMEM, s>>>(tq, tk, tv, tg, tdy, tH, ka);
            rc = launch_status();
        }
    }
    if (rc == LIZARD_OK && gqa_bytes) rc = launch_gqa_reduce<__nv_bfloat16, DH>(bg, ba.dk, ba.dv, s);
    if (cudaFreeAsync(scratch, s) != cudaSuccess && rc == LIZARD_OK) rc = LIZARD_ERR_CUDA;
    return rc;
}

// [rows][K] bf16 row-major as a 3-D tensor {K, rows, 1}; 64 x box_rows
// boxes, 128B swizzle, rows and columns past the end read as zero.
static bool make_rows_map(CUtensorMap *map, const void *base, int rows, int K, int box_rows)
{
    encode_tiled_fn enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)K, (cuuint64_t)rows, 1};
    cuuint64_t strides[2] = {(cuuint64_t)K * 2, (cuuint64_t)rows * K * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ---------------------------------------------------------------- allocation-free prefill
// Segment states of lizard_attn_prefill_noalloc: a fixed array in device
// memory, held by every GPU that loads this library until the process ends.
constexpr size_t NOALLOC_FLOATS = LIZARD_NOALLOC_SCRATCH_BYTES / sizeof(float);
static __device__ __align__(256) float g_prefill_scratch[NOALLOC_FLOATS];

// The driver's cuCtxGetCurrent, looked up once (as the tensor-map encoder).
typedef CUresult (*ctx_get_current_fn)(CUcontext *);
static ctx_get_current_fn lookup_ctx_get_current()
{
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
        return reinterpret_cast<ctx_get_current_fn>(p);
    return nullptr;
}
static CUcontext current_context()
{
    static const ctx_get_current_fn fn = lookup_ctx_get_current();
    CUcontext c = nullptr;
    if (!fn || fn(&c) != CUDA_SUCCESS) return nullptr;
    return c;
}

// The array's device address on the current device.  In host code the name
// g_prefill_scratch is a host-side stand-in, not a device address, so it is
// looked up (cudaGetSymbolAddress) with the device current, once per device
// and context: a device reset gives the device a new context in which the
// module, and so the array, is loaded again, and the lookup is repeated.
static lizard_status noalloc_scratch(float **out)
{
    constexpr int MAX_DEV = 64;
    static std::mutex mu;
    static float *addr[MAX_DEV] = {};
    static CUcontext ctx[MAX_DEV] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEV) return LIZARD_ERR_CUDA;
    std::lock_guard<std::mutex> lock(mu);
    const CUcontext now = current_context();
    if (!addr[dev] || !now || now != ctx[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_prefill_scratch) != cudaSuccess || !p) return LIZARD_ERR_CUDA;
        addr[dev] = static_cast<float *>(p);
        ctx[dev] = current_context();  // the lookup makes the device's context current
    }
    *out = addr[dev];
    return LIZARD_OK;
}

}  // namespace lizard

using namespace lizard;

extern "C" {

const char *lizard_status_string(lizard_status s)
{
    switch (s) {
    case LIZARD_OK: return "LIZARD_OK";
    case LIZARD_ERR_INVALID_ARG: return "LIZARD_ERR_INVALID_ARG";
    case LIZARD_ERR_UNSUPPORTED: return "LIZARD_ERR_UNSUPPORTED";
    case LIZARD_ERR_CUDA: return "LIZARD_ERR_CUDA";
    case LIZARD_ERR_TIMEOUT: return "LIZARD_ERR_TIMEOUT";
    }
    return "LIZARD_ERR_UNKNOWN";
}

lizard_status lizard_state_init(const lizard_state *st, lizard_stream_t stream)
{
    lizard_status rc = check_state(st);
    if (rc != LIZARD_OK) return rc;
    const size_t nS = (size_t)st->B * st->H * st->dk * st->dv;
    const size_t ring_bytes = (size_t)st->B * st->H * st->w * st->dk * esize(st->dtype);
    if (st->B == 0) return LIZARD_OK;
    int blocks = (int)((nS / 4 + 255) / 256);
    if (blocks > 148 * 16) blocks = 148 * 16;
    state_init_kernel<<<blocks, 256, 0, (cudaStream_t)stream>>>(
        st->S, nS, static_cast<uint4 *>(st->ring_k), static_cast<uint4 *>(st->ring_v), ring_bytes / 16, st->pos,
        st->B);
    return launch_status();
}

// A variant's key/value grouping and per-head weights, validated.
static lizard_status variant_of(const lizard_variant *var, int H, int *group, const float **alpha_h)
{
    *group = 1;
    *alpha_h = nullptr;
    if (!var) return LIZARD_OK;
    const int Hkv = var->Hkv == 0 ? H : var->Hkv;
    if (Hkv < 1 || Hkv > H || H % Hkv != 0) return LIZARD_ERR_INVALID_ARG;
    if (var->alpha_h && (reinterpret_cast<uintptr_t>(var->alpha_h) & 3u)) return LIZARD_ERR_INVALID_ARG;
    *group = H / Hkv;
    *alpha_h = var->alpha_h;
    return LIZARD_OK;
}

lizard_status lizard_attn_prefill(const void *q, const void *k, const void *v, const void *g, const void *meta_k,
                                  float alpha, int B, int H, int L, int dk, int dv, int w, int m,
                                  lizard_dtype dtype, void *y, const lizard_state *st, lizard_stream_t stream)
{
    return lizard_attn_prefill_v(q, k, v, g, meta_k, alpha, B, H, L, dk, dv, w, m, dtype, y, st, nullptr, stream);
}

lizard_status lizard_attn_prefill_v(const void *q, const void *k, const void *v, const void *g, const void *meta_k,
                                    float alpha, int B, int H, int L, int dk, int dv, int w, int m,
                                    lizard_dtype dtype, void *y, const lizard_state *st, const lizard_variant *var,
                                    lizard_stream_t stream)
{
    if (!dtype_ok(dtype)) return LIZARD_ERR_INVALID_ARG;
    if (B < 0 || H < 1 || L < 0 || dk < 1 || dv < 1 || w < 1 || m < 0) return LIZARD_ERR_INVALID_ARG;
    int group = 1;
    const float *alpha_h = nullptr;
    lizard_status vrc = variant_of(var, H, &group, &alpha_h);
    if (vrc != LIZARD_OK) return vrc;
    // An empty prompt (L == 0) has no token tensors to point at.
    if (L > 0 && (!q || !k || !v || !g || !y)) return LIZARD_ERR_INVALID_ARG;
    if (m > 0 && !meta_k) return LIZARD_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(g) || !aligned16(y) ||
        (m > 0 && !aligned16(meta_k)))
        return LIZARD_ERR_INVALID_ARG;
    if (dk != dv || (dk != 64 && dk != 128 && dk != 256)) return LIZARD_ERR_UNSUPPORTED;
    if (w > LIZARD_MAX_WINDOW || m > LIZARD_MAX_META) return LIZARD_ERR_UNSUPPORTED;
    if ((int64_t)B * H > 2147483647LL || (int64_t)L * dk > (int64_t)1 << 40) return LIZARD_ERR_UNSUPPORTED;
    if (st) {
        lizard_status rc = check_state(st);
        if (rc != LIZARD_OK) return rc;
        if (st->B != B || st->H != H || st->dk != dk || st->dv != dv || st->w != w || st->dtype != dtype)
            return LIZARD_ERR_INVALID_ARG;
    }
    if (B == 0) return LIZARD_OK;
    if (L == 0) return st ? lizard_state_init(st, stream) : LIZARD_OK;  // the empty prompt leaves the empty state
    PrefillArgs pa{q, k, v, g, meta_k, y, alpha, B, H, L, w, m,
                   st ? st->S : nullptr, st ? st->ring_k : nullptr, st ? st->ring_v : nullptr,
                   st ? st->pos : nullptr, 0, nullptr, alpha_h, group};
    cudaStream_t s = (cudaStream_t)stream;
    if (dk == 256)  // CUDA cores, value slices
        return dtype == LIZARD_BF16 ? launch_prefill<__nv_bfloat16, 256>(pa, s) : launch_prefill<float, 256>(pa, s);
    if (dtype == LIZARD_BF16)
        return dk == 128 ? launch_prefill_ws(pa, s)
                         : launch_prefill_ws(pa, s, nullptr, 0, 0, 64);
    return dk == 128 ? launch_prefill<float, 128>(pa, s) : launch_prefill<float, 64>(pa, s);
}

lizard_status lizard_attn_prefill_noalloc(const void *q, const void *k, const void *v, const void *g,
                                          const void *meta_k, float alpha, int B, int H, int L, int dk, int dv, int w,
                                          int m, lizard_dtype dtype, void *y, const lizard_state *st,
                                          lizard_stream_t stream)
{
    if (!dtype_ok(dtype)) return LIZARD_ERR_INVALID_ARG;
    if (B < 0 || H < 1 || L < 0 || dk < 1 || dv < 1 || w < 1 || m < 0) return LIZARD_ERR_INVALID_ARG;
    if (L > 0 && (!q || !k || !v || !g || !y)) return LIZARD_ERR_INVALID_ARG;
    if (m > 0 && !meta_k) return LIZARD_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(g) || !aligned16(y) ||
        (m > 0 && !aligned16(meta_k)))
        return LIZARD_ERR_INVALID_ARG;
    // The variant covers the tensor-core prefill, the one with scratch.
    if (dtype != LIZARD_BF16 || dk != dv || !(dk == 128 || dk == 64) || w > LIZARD_MAX_WINDOW ||
        m > LIZARD_MAX_META)
        return LIZARD_ERR_UNSUPPORTED;
    if ((int64_t)B * H > 2147483647LL || (int64_t)L * dk > (int64_t)1 << 40) return LIZARD_ERR_UNSUPPORTED;
    if (st) {
        lizard_status rc = check_state(st);
        if (rc != LIZARD_OK) return rc;
        if (st->B != B || st->H != H || st->dk != dk || st->dv != dv || st->w != w || st->dtype != dtype)
            return LIZARD_ERR_INVALID_ARG;
    }
    if (B == 0) return LIZARD_OK;
    if (L == 0) return st ? lizard_state_init(st, stream) : LIZARD_OK;
    float *scratch = nullptr;
    lizard_status rc = noalloc_scratch(&scratch);
    if (rc != LIZARD_OK) return rc;
    PrefillArgs pa{q, k, v, g, meta_k, y, alpha, B, H, L, w, m,
                   st ? st->S : nullptr, st ? st->ring_k : nullptr, st ? st->ring_v : nullptr,
                   st ? st->pos : nullptr, 0, nullptr, nullptr, 1};
    // Segment states beyond LIZARD_NOALLOC_SCRATCH_BYTES: LIZARD_ERR_UNSUPPORTED, nothing launched.
    return launch_prefill_ws(pa, (cudaStream_t)stream, scratch, LIZARD_NOALLOC_SCRATCH_BYTES, 0, dk);
}

lizard_status lizard_attn_prefill_continue(const void *q, const void *k, const void *v, const void *g,
                                          const void *meta_k, float alpha, int L, int m, void *y,
                                          const lizard_state *st, lizard_stream_t stream)
{
    return lizard_attn_prefill_continue_v(q, k, v, g, meta_k, alpha, L, m, y, st, nullptr, stream);
}

lizard_status lizard_attn_prefill_continue_v(const void *q, const void *k, const void *v, const void *g,
                                            const void *meta_k, float alpha, int L, int m, void *y,
                                            const lizard_state *st, const lizard_variant *var, lizard_stream_t stream)
{
    lizard_status rc = check_state(st);
    if (rc != LIZARD_OK) return rc;
    int group = 1;
    const float *alpha_h = nullptr;
    rc = variant_of(var, st->H, &group, &alpha_h);
    if (rc != LIZARD_OK) return rc;
    if (L < 0 || m < 0) return LIZARD_ERR_INVALID_ARG;
    if (L > 0 && (!q || !k || !v || !g || !y)) return LIZARD_ERR_INVALID_ARG;
    if (m > 0 && !meta_k) return LIZARD_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(g) || !aligned16(y) ||
        (m > 0 && !aligned16(meta_k)))
        return LIZARD_ERR_INVALID_ARG;
    if (m > LIZARD_MAX_META) return LIZARD_ERR_UNSUPPORTED;
    const int B = st->B, H = st->H, dk = st->dk, w = st->w;
    if ((int64_t)B * H > 2147483647LL || (int64_t)L * dk > (int64_t)1 << 40) return LIZARD_ERR_UNSUPPORTED;
    // The CTAs of one sequence count their arrivals in pos's high bits
    // (H x segments of at most the SM count must stay below 2^23).
    if (H > 16384) return LIZARD_ERR_UNSUPPORTED;
    if (B == 0 || L == 0) return LIZARD_OK;  // no new token: the state stays as it is
    PrefillArgs pa{q, k, v, g, meta_k, y, alpha, B, H, L, w, m, st->S, st->ring_k, st->ring_v, st->pos, 1, st->S,
                   alpha_h, group};
    cudaStream_t s = (cudaStream_t)stream;
    if (dk == 256)  // CUDA cores, value slices
        return st->dtype == LIZARD_BF16 ? launch_prefill<__nv_bfloat16, 256>(pa, s) : launch_prefill<float, 256>(pa, s);
    if (st->dtype == LIZARD_BF16)
        return dk == 128 ? launch_prefill_ws(pa, s)
                         : launch_prefill_ws(pa, s, nullptr, 0, 0, 64);
    return dk == 128 ? launch_prefill<float, 128>(pa, s) : launch_prefill<float, 64>(pa, s);
}

lizard_status lizard_attn_backward(const void *q, const void *k, const void *v, const void *g, const void *meta_k,
                                   float alpha, int B, int H, int L, int dk, int dv, int w, int m, lizard_dtype dtype,
                                   const void *dy, void *dq, void *dk_out, void *dv_out, void *dg, float *dmeta_k,
                                   float *dalpha, lizard_stream_t stream)
{
    return lizard_attn_backward_v(q, k, v, g, meta_k, alpha, B, H, L, dk, dv, w, m, dtype, dy, dq, dk_out, dv_out, dg,
                                  dmeta_k, dalpha, nullptr, stream);
}

lizard_status lizard_attn_backward_v(const void *q, const void *k, const void *v, const void *g, const void *meta_k,
                                     float alpha, int B, int H, int L, int dk, int dv, int w, int m, lizard_dtype dtype,
                                     const void *dy, void *dq, void *dk_out, void *dv_out, void *dg, float *dmeta_k,
                                     float *dalpha, const lizard_variant *var, lizard_stream_t stream)
{
    if (!dtype_ok(dtype)) return LIZARD_ERR_INVALID_ARG;
    if (B < 0 || H < 1 || L < 0 || dk < 1 || dv < 1 || w < 1 || m < 0) return LIZARD_ERR_INVALID_ARG;
    int group = 1;
    const float *alpha_h = nullptr;
    lizard_status vrc = variant_of(var, H, &group, &alpha_h);
    if (vrc != LIZARD_OK) return vrc;
    if (L > 0 && B > 0 && (!q || !k || !v || !g || !dy || !dq || !dk_out || !dv_out || !dg))
        return LIZARD_ERR_INVALID_ARG;
    if (m > 0 && (!meta_k || !dmeta_k)) return LIZARD_ERR_INVALID_ARG;
    if (!dalpha || (reinterpret_cast<uintptr_t>(dalpha) & 3u)) return LIZARD_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(g) || !aligned16(dy) || !aligned16(dq) ||
        !aligned16(dk_out) || !aligned16(dv_out) || !aligned16(dg) || (m > 0 && (!aligned16(meta_k) || !aligned16(dmeta_k))))
        return LIZARD_ERR_INVALID_ARG;
    if (dk != dv || (dk != 64 && dk != 128)) return LIZARD_ERR_UNSUPPORTED;
    if (w > LIZARD_MAX_WINDOW || m > LIZARD_MAX_META) return LIZARD_ERR_UNSUPPORTED;
    if ((int64_t)B * H > 2147483647LL || (int64_t)L * dk > (int64_t)1 << 40) return LIZARD_ERR_UNSUPPORTED;
    cudaStream_t s = (cudaStream_t)stream;
    if (B == 0 || L == 0) {  // no token: the parameter gradients are zero
        if (cudaMemsetAsync(dalpha, 0, sizeof(float) * (alpha_h ? H : 1), s) != cudaSuccess) return LIZARD_ERR_CUDA;
        if (m > 0 && cudaMemsetAsync(dmeta_k, 0, sizeof(float) * H * m * dk, s) != cudaSuccess) return LIZARD_ERR_CUDA;
        return LIZARD_OK;
    }
    BackwardArgs ba{q, k, v, g, meta_k, dy, dq, dk_out, dv_out, dg, alpha, B, H, L, w, m,
                    nullptr, nullptr, nullptr, nullptr, nullptr, alpha_h, group};
    float *dmu = m > 0 ? dmeta_k : nullptr;
    if (dtype == LIZARD_BF16 && w <= 65)
        return dk == 128 ? launch_backward_tc<128>(ba, dmu, dalpha, s) : launch_backward_tc<64>(ba, dmu, dalpha, s);
    if (dtype == LIZARD_BF16)
        return dk == 128 ? launch_backward<__nv_bfloat16, 128>(ba, dmu, dalpha, s)
                         : launch_backward<__nv_bfloat16, 64>(ba, dmu, dalpha, s);
    return dk == 128 ? launch_backward<float, 128>(ba, dmu, dalpha, s) : launch_backward<float, 64>(ba, dmu, dalpha, s);
}

lizard_status lizard_gate_projection(const void *x, const void *w_gamma, int B, int L, int dmodel, int H, int dk,
                                    lizard_dtype dtype, void *g, lizard_stream_t stream)
{
    if (!dtype_ok(dtype)) return LIZARD_ERR_INVALID_ARG;
    if (B < 0 || L < 0 || dmodel < 1 || H < 1 || dk < 1) return LIZARD_ERR_INVALID_ARG;
    const int64_t M = (int64_t)B * L;
    if (M > 0 && (!x || !w_gamma || !g)) return LIZARD_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(w_gamma) || !aligned16(g)) return LIZARD_ERR_INVALID_ARG;
    if (dtype != LIZARD_BF16 || dk != gproj::DK || dmodel % 8 != 0) return LIZARD_ERR_UNSUPPORTED;
    if (M > 2147483647LL || (int64_t)H * dk > 2147483647LL || M * dmodel > ((int64_t)1 << 40))
        return LIZARD_ERR_UNSUPPORTED;
    if (M == 0) return LIZARD_OK;
    // two heads per tile when the head count allows it
    const int nh = H % 2 == 0 ? 2 : 1;
    CUtensorMap tx, tw;
    if (!make_rows_map(&tx, x, (int)M, dmodel, gproj::BM) || !make_rows_map(&tw, w_gamma, H * dk, dmodel, gproj::DK * nh))
        return LIZARD_ERR_CUDA;
    const int64_t tiles = ((M + gproj::BM - 1) / gproj::BM) * (H / nh);
    if (tiles > 2147483647LL) return LIZARD_ERR_UNSUPPORTED;
    gproj::Args ga{static_cast<__nv_bfloat16 *>(g), (int)M, dmodel, L, H};
    auto kern = nh == 2 ? gproj::gate_proj_kernel<2> : gproj::gate_proj_kernel<1>;
    const uint32_t smem = nh == 2 ? gproj::Cfg<2>::SMEM : gproj::Cfg<1>::SMEM;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return LIZARD_ERR_CUDA;
    const int64_t ctas = tiles < sm_count() ? tiles : sm_count();  // persistent: one CTA per SM
    kern<<<(unsigned)ctas, gproj::THREADS, smem, (cudaStream_t)stream>>>(tx, tw, ga);
    return launch_status();
}

lizard_status lizard_attn_decode_step(const void *q, const void *k, const void *v, const void *g, const void *meta_k,
                                      float alpha, int m, void *y, const lizard_state *st, lizard_stream_t stream)
{
    return lizard_attn_decode_step_v(q, k, v, g, meta_k, alpha, m, y, st, nullptr, stream);
}

lizard_status lizard_attn_decode_step_v(const void *q, const void *k, const void *v, const void *g,
                                        const void *meta_k, float alpha, int m, void *y, const lizard_state *st,
                                        const lizard_variant *var, lizard_stream_t stream)
{
    lizard_status rc = check_state(st);
    if (rc != LIZARD_OK) return rc;
    int group = 1;
    const float *alpha_h = nullptr;
    rc = variant_of(var, st->H, &group, &alpha_h);
    if (rc != LIZARD_OK) return rc;
    if (m < 0) return LIZARD_ERR_INVALID_ARG;
    if (!q || !k || !v || !g || !y || (m > 0 && !meta_k)) return LIZARD_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(g) || !aligned16(y) ||
        (m > 0 && !aligned16(meta_k)))
        return LIZARD_ERR_INVALID_ARG;
    if (m > LIZARD_MAX_META) return LIZARD_ERR_UNSUPPORTED;
    // The CTAs of one sequence (up to 8 H) count their arrivals in pos's
    // high bits, which hold counts below 2^23.
    if (st->H >= (1 << 20)) return LIZARD_ERR_UNSUPPORTED;
    if (st->B == 0) return LIZARD_OK;
    DecodeArgs da{q, k, v, g, meta_k, y, st->S, st->ring_k, st->ring_v, st->pos, alpha, st->B, st->H, st->w, m,
                  alpha_h, group, -1};
    cudaStream_t s = (cudaStream_t)stream;
    if (st->dtype == LIZARD_BF16)
        return st->dk == 256   ? launch_decode<__nv_bfloat16, 256>(da, s)
               : st->dk == 128 ? launch_decode<__nv_bfloat16, 128>(da, s)
                               : launch_decode<__nv_bfloat16, 64>(da, s);
    return st->dk == 256 ? launch_decode<float, 256>(da, s)
           : st->dk == 128 ? launch_decode<float, 128>(da, s)
                           : launch_decode<float, 64>(da, s);
}

lizard_status lizard_scratch_trim(size_t keep_bytes)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return LIZARD_ERR_CUDA;
    cudaMemPool_t pool;
    if (scratch_pool(dev, false, &pool) != cudaSuccess) return LIZARD_ERR_CUDA;
    if (!pool) return LIZARD_OK;
    return cudaMemPoolTrimTo(pool, keep_bytes) == cudaSuccess ? LIZARD_OK : LIZARD_ERR_CUDA;
}

lizard_status lizard_scratch_reserved(size_t *bytes)
{
    if (!bytes) return LIZARD_ERR_INVALID_ARG;
    *bytes = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return LIZARD_ERR_CUDA;
    cudaMemPool_t pool;
    if (scratch_pool(dev, false, &pool) != cudaSuccess) return LIZARD_ERR_CUDA;
    if (!pool) return LIZARD_OK;
    uint64_t v = 0;
    if (cudaMemPoolGetAttribute(pool, cudaMemPoolAttrReservedMemCurrent, &v) != cudaSuccess) return LIZARD_ERR_CUDA;
    *bytes = (size_t)v;
    return LIZARD_OK;
}

lizard_status lizard_check_device_status(lizard_stream_t stream)
{
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return LIZARD_ERR_CUDA;
    int word = DEV_OK, zero = DEV_OK;
    if (cudaMemcpyFromSymbol(&word, g_device_error, sizeof word) != cudaSuccess) return LIZARD_ERR_CUDA;
    if (word != DEV_OK && cudaMemcpyToSymbol(g_device_error, &zero, sizeof zero) != cudaSuccess)
        return LIZARD_ERR_CUDA;
    if (word == DEV_OK) return LIZARD_OK;
    return word == DEV_BAD_POS ? LIZARD_ERR_INVALID_ARG : LIZARD_ERR_TIMEOUT;
}

#ifdef LIZARD_TRACE
// Debug builds only: the clock trace of the warp-specialised prefill's CTA 0.
__attribute__((visibility("default"))) int lizard_debug_trace(unsigned long long *out)
{
    return cudaMemcpyFromSymbol(out, ws::g_ws_trace, sizeof(ws::g_ws_trace)) == cudaSuccess ? 0 : 1;
}
#endif

}  // extern "C"
