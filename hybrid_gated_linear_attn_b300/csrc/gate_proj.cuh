// gate_proj.cuh -- the gate projection ahead of the operator on tcgen05:
// g[b][h][t][i] = sum_c x[b][t][c] W[h dk + i][c]  (bf16 in, fp32 accumulate,
// bf16 out), written straight into the operator's head-major layout.
//
// Lizard (gist.science/de section 2 item 1): the gate Gamma = sigmoid(W_gamma x)
// decides how much of the past each key dimension keeps; the operator takes
// its logits g = W_gamma x (and applies the log-sigmoid itself).
//
// Output tiles of 128 x (128 NH) (128 tokens x NH heads of dk = 128; NH = 2
// when the head count is even, which cuts the operand bytes per flop by a
// quarter); consecutive tiles sweep the heads of one token block (the x
// block and all of W stay in L2).  One persistent CTA per SM walks its
// tiles: a four-stage TMA pipeline feeds 64-wide K slices (128B-swizzled,
// K-major) to one MMA-issuing thread; two fp32 accumulators in tensor
// memory alternate between tiles, so four epilogue warps convert and store
// each token's 128 outputs (256 contiguous bytes) of one tile while the next
// tile's products run.  Every wait is bounded: a
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
    static constexpr uint32_t SMEM = OFF_BAR + (2 * STAGES + 5) * 8 + 16 + 1024;
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

// Persistent: grid = min(tiles, SMs) CTAs; CTA i takes tiles i, i + grid,
// ...  Tile index -> heads NH (tile % (H / NH)) .. + NH - 1, token block
// tile / (H / NH).  Two accumulators in tensor memory: the products of a
// tile go into one while the epilogue drains the other, so the epilogue
// overlaps the next tile's main loop.  tw's box is BN rows high.
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
    uint64_t *full = reinterpret_cast<uint64_t *>(sm + OFF_BAR), *empty = full + STAGES;
    uint64_t *acc_full = empty + STAGES, *acc_empty = acc_full + 2, *done = acc_empty + 2;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(done + 1);
    volatile int *abort_f = reinterpret_cast<volatile int *>(tslot + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int HT = a.H / NH;
    const int tiles = (a.M + BM - 1) / BM * HT;
    const int KT = (a.K + BK - 1) / BK;

    if (warp == 1) {
        tmem_alloc(tslot, 2 * BN);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&acc_full[i], 1);
            mbar_init(&acc_empty[i], 1);
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
    auto give_up = [&]() {
        *abort_f = 1;
        atomicExch(&g_device_error, DEV_TIMEOUT);
    };

    if (warp == 0) {
        if (lane == 0) {  // producer: one k-slice count over all of this CTA's tiles
            uint32_t g = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < tiles && ok; tile += gridDim.x) {
                const int m0 = (tile / HT) * BM, n0 = (tile % HT) * NH * DK;
                for (int kt = 0; kt < KT; ++kt, ++g) {
                    const uint32_t s = g % STAGES;
                    if (g >= STAGES && !wait_bar(&empty[s], g / STAGES - 1, abort_f)) {
                        give_up();
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&full[s], STAGE);
                    tma_load_3d(sm + s * STAGE, &tx, &full[s], kt * BK, m0, 0);
                    tma_load_3d(sm + s * STAGE + A_BYTES, &tw, &full[s], kt * BK, n0, 0);
                }
            }
            // drain: the copies in flight land before shared memory is released
            for (uint32_t u = g > STAGES ? g - STAGES : 0; u < g; ++u)
                wait_bar(&full[u % STAGES], u / STAGES, abort_f);
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {  // MMA issuer
            const uint32_t id = instr_desc(BM, BN, FMT_BF16, 0, 0);
            uint32_t g = 0;
            int li = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < tiles && ok; tile += gridDim.x, ++li) {
                const int acc = li & 1;
                // the epilogue has drained this accumulator (two tiles ago)
                if (li >= 2 && !wait_bar(&acc_empty[acc], (li >> 1) - 1, abort_f)) {
                    give_up();
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem + acc * BN;
                for (int kt = 0; kt < KT; ++kt, ++g) {
                    const uint32_t s = g % STAGES;
                    if (!wait_bar(&full[s], g / STAGES, abort_f)) {
                        give_up();
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t ab = sb + s * STAGE, bb = ab + A_BYTES;
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        mma_bf16_ss(d, smem_desc(ab + kk * 32, 16, 1024), smem_desc(bb + kk * 32, 16, 1024), id,
                                    (kt > 0 || kk > 0) ? 1u : 0u);
                    mma_commit(&empty[s]);
                }
                if (ok) mma_commit(&acc_full[acc]);
            }
            mma_commit(done);
            wait_bar(done, 0, abort_f);  // every product is done before tensor memory is released
        }
        __syncwarp();
    } else if (warp >= 4) {
        // epilogue: thread = one token row of the tile (tensor-memory lane)
        const int q = warp & 3, row = 32 * q + lane;
        int li = 0;
        for (int tile = blockIdx.x; tile < tiles; tile += gridDim.x, ++li) {
            const int acc = li & 1;
            bool ok = true;
            if (lane == 0) ok = wait_bar(&acc_full[acc], li >> 1, abort_f);
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            if (!ok) {
                if (lane == 0) give_up();
                break;
            }
            tc_fence_after();
            const int h0 = (tile % HT) * NH, m = (tile / HT) * BM + row;
            const int b = m / a.L, t = m % a.L;
            const uint32_t src = tmem + acc * BN + ((uint32_t)(32 * q) << 16);
#pragma unroll 1
            for (int cc = 0; cc < BN; cc += 16) {
                uint4 *dst = reinterpret_cast<uint4 *>(a.g + (((size_t)b * a.H + h0 + cc / DK) * a.L + t) * DK);
                uint32_t r[16];
                tmem_ld16(src + cc, r);
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
            // the accumulator is read: the issuer may start the tile after next in it
            tc_fence_before();
            asm volatile("bar.sync 1, 128;" ::: "memory");  // the four epilogue warps
            if (warp == 4 && lane == 0) mbar_arrive(&acc_empty[acc]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, 2 * BN);
}

}  // namespace gproj
}  // namespace lizard
