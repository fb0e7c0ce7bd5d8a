// gate_proj.cuh -- the gate projection ahead of the operator on tcgen05:
// g[b][h][t][i] = sum_c x[b][t][c] W[h dk + i][c]  (bf16 in, fp32 accumulate,
// bf16 out), written straight into the operator's head-major layout.
//
// Lizard (gist.science/de section 2 item 1): the gate Gamma = sigmoid(W_gamma x)
// decides how much of the past each key dimension keeps; the operator takes
// its logits g = W_gamma x (and applies the log-sigmoid itself).
//
// One CTA per 128 x (128 NH) output tile (128 tokens x NH heads of dk =
// 128; NH = 2 when the head count is even, which cuts the operand bytes per
// flop by a quarter), consecutive CTAs sweeping the heads of one token block
// (the x block and all of W stay in L2).  A four-stage TMA pipeline feeds 64-wide K slices
// (128B-swizzled, K-major) to one MMA-issuing thread; the fp32 accumulator
// lives in tensor memory; four epilogue warps convert and store each
// token's 128 outputs (256 contiguous bytes).  Every wait is bounded: a
// timeout records DEV_TIMEOUT, drains what is in flight and returns.
#pragma once

#include "common.cuh"
#include "sm100.cuh"

namespace lizard {
namespace gproj {

using namespace sm100;

constexpr int BM = 128, DK = 128, BK = 64;
constexpr int STAGES = 4;
constexpr int THREADS = 256;
constexpr uint32_t WAIT = 1u << 21;
template <int NH>
struct Cfg {
    static constexpr int BN = DK * NH;
    static constexpr uint32_t A_BYTES = BM * BK * 2, B_BYTES = BN * BK * 2;
    static constexpr uint32_t STAGE = A_BYTES + B_BYTES;
    static constexpr uint32_t OFF_BAR = STAGES * STAGE;
    static constexpr uint32_t SMEM = OFF_BAR + (2 * STAGES + 1) * 8 + 16 + 1024;
    static_assert(SMEM <= 232448, "shared memory budget");
};

struct Args {
    __nv_bfloat16 *g;  // [B][H][L][DK]
    int M, K, L, H;    // M = B * L tokens, K = dmodel
};

__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t use, volatile int *abort_f)
{
    for (uint32_t i = 0; i < WAIT; ++i) {
        if (mbar_try_wait(bar, use & 1u)) return true;
        if ((i & 255u) == 255u && *abort_f) return false;
    }
    return false;
}

// grid = ceil(M / BM) * (H / NH): tile = blockIdx.x, heads NH (tile % (H / NH))
// .. + NH - 1, token block = tile / (H / NH).  tw's box is BN rows high.
template <int NH>
__global__ void __launch_bounds__(THREADS, 1)
    gate_proj_kernel(const __grid_constant__ CUtensorMap tx, const __grid_constant__ CUtensorMap tw, const Args a)
{
    using G = Cfg<NH>;
    constexpr int BN = G::BN;
    constexpr uint32_t A_BYTES = G::A_BYTES, STAGE = G::STAGE, OFF_BAR = G::OFF_BAR;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = smem_align1024(smem_raw);
    const uint32_t sb = smem_u32(sm);
    uint64_t *full = reinterpret_cast<uint64_t *>(sm + OFF_BAR), *empty = full + STAGES, *done = empty + STAGES;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(done + 1);
    volatile int *abort_f = reinterpret_cast<volatile int *>(tslot + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int HT = a.H / NH;
    const int h0 = (blockIdx.x % HT) * NH, m0 = (blockIdx.x / HT) * BM, n0 = h0 * DK;
    const int KT = (a.K + BK - 1) / BK;

    if (warp == 1) {
        tmem_alloc(tslot, BN);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(done, 1);
        *abort_f = 0;
        fence_mbar_init();
        prefetch_tmap(&tx);
        prefetch_tmap(&tw);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    bool failed = false;
    auto give_up = [&]() {
        failed = true;
        *abort_f = 1;
        atomicExch(&g_device_error, DEV_TIMEOUT);
    };

    if (warp == 0) {
        if (lane == 0) {  // producer
            uint32_t issued = 0;
            for (int kt = 0; kt < KT; ++kt) {
                const int s = kt % STAGES;
                if (kt >= STAGES && !wait_bar(&empty[s], kt / STAGES - 1, abort_f)) { give_up(); break; }
                mbar_arrive_expect_tx(&full[s], STAGE);
                tma_load_3d(sm + s * STAGE, &tx, &full[s], kt * BK, m0, 0);
                tma_load_3d(sm + s * STAGE + A_BYTES, &tw, &full[s], kt * BK, n0, 0);
                ++issued;
            }
            // drain: the copies in flight land before shared memory is released
            for (uint32_t u = issued > STAGES ? issued - STAGES : 0; u < issued; ++u)
                wait_bar(&full[u % STAGES], u / STAGES, abort_f);
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {  // MMA issuer
            const uint32_t id = instr_desc(BM, BN, FMT_BF16, 0, 0);
            for (int kt = 0; kt < KT; ++kt) {
                const int s = kt % STAGES;
                if (!wait_bar(&full[s], kt / STAGES, abort_f)) { give_up(); break; }
                tc_fence_after();
                const uint32_t ab = sb + s * STAGE, bb = ab + A_BYTES;
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk)
                    mma_bf16_ss(tmem, smem_desc(ab + kk * 32, 16, 1024), smem_desc(bb + kk * 32, 16, 1024), id,
                                (kt > 0 || kk > 0) ? 1u : 0u);
                mma_commit(&empty[s]);
            }
            mma_commit(done);
            wait_bar(done, 0, abort_f);  // every product is done before tensor memory is released
        }
        __syncwarp();
    } else if (warp >= 4) {
        // epilogue: thread = one token row of the tile (tensor-memory lane)
        const int q = warp & 3, row = 32 * q + lane, m = m0 + row;
        bool ok = true;
        if (lane == 0) ok = wait_bar(done, 0, abort_f);
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) {
            if (lane == 0) give_up();
        } else {
            tc_fence_after();
            const int b = m / a.L, t = m % a.L;
#pragma unroll 1
            for (int cc = 0; cc < BN; cc += 16) {
                uint4 *dst = reinterpret_cast<uint4 *>(a.g + (((size_t)b * a.H + h0 + cc / DK) * a.L + t) * DK);
                uint32_t r[16];
                tmem_ld16(tmem + ((uint32_t)(32 * q) << 16) + cc, r);
                tmem_wait_ld();
                uint32_t pk[8];
#pragma unroll
                for (int e = 0; e < 16; e += 2) {
                    __nv_bfloat162 v2 = __floats2bfloat162_rn(__uint_as_float(r[e]), __uint_as_float(r[e + 1]));
                    pk[e / 2] = *reinterpret_cast<uint32_t *>(&v2);
                }
                if (m < a.M) {
                    dst[(cc % DK) / 8] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                    dst[(cc % DK) / 8 + 1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
                }
            }
        }
    }
    (void)failed;
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, BN);
}

}  // namespace gproj
}  // namespace lizard
