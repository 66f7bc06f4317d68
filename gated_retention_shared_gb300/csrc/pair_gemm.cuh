// pair_gemm.cuh -- persistent bf16 GEMM  Y[R, ncols] = X[R, dm] W[dm, ncols]  on
// CTA pairs (a cluster of two, one CTA per SM), fp32 accumulate in tensor memory,
// with the epilogue left to the caller.  Used by the projections that produce the
// attention inputs: the shared K^/V^ projection and the gated-retention layer's
// q/k/v/gate projection.
//
// Tiles are 256 rows x 256 columns.  The even CTA issues tcgen05.mma.cta_group::2
// of shape 256 x 256 x 16; each CTA stages its own 128 rows of X (K-major) and its
// own 128 of the 256 W columns (N-major) per 64-deep step, 32 KB in a 6-stage TMA
// ring with 128-byte swizzle, and the MMA reads the other half from the peer's
// shared memory.  Each CTA's tensor memory holds its 128 rows x 256 columns in one
// of two accumulators (512 columns), so one tile drains while the next one runs.
//   * both CTAs' copies of a stage complete on the even CTA's `full` barrier, whose
//     one arrival (the even producer's) expects the 64 KB of both; a peer copy that
//     lands before that arrival leaves the phase pending, and the odd producer
//     refills a stage only after the MMA freed it, i.e. after the phase;
//   * the even CTA's MMA commit frees the stage in both CTAs (`empty`, multicast)
//     and announces a finished accumulator to both epilogues (`acc_full`);
//   * both epilogues hand the accumulator back on the even CTA's `acc_empty`.
// Warps: 0 TMA producer, 1 MMA issuer (even CTA), 2-5 epilogue (thread = row).
// Rows and columns past the matrices arrive zero-filled; the epilogue skips rows
// past R and 32-column blocks past ncols.  Every wait is bounded: a timeout records
// kErrMagic | code (codes code0 .. code0 + 3) in *err and unwinds.
#pragma once

#include "common.cuh"
#include "tc.cuh"

namespace yoco {

namespace pairgemm {

using namespace tc;

constexpr int kM = 256, kN = 256, kK = 64, kStages = 6, kThreads = 192;
constexpr int kAtile = 128 * kK * 2;      // 16 KB: this CTA's 128 rows of X
constexpr int kBtile = kK * 128 * 2;      // 16 KB: this CTA's 128 columns of W
constexpr int kStage = kAtile + kBtile;   // 32 KB

struct Smem {
    uint64_t full[kStages], empty[kStages];
    uint64_t acc_full[2], acc_empty[2], drain;
    uint32_t tmem_base;
    int abort_flag;
    int go;
};

constexpr size_t kSmemBytes = (size_t)kStages * kStage + 1024 + sizeof(Smem);
static_assert(kSmemBytes <= 232448, "pair tiles and control block must fit shared memory");

// Kernel body.  `wload(dst, bar, col, k0)` issues the TMA load (tma_load_2d_pair)
// of the 64 x 64 W block whose first column is `col` and first row `k0`.
// `epi(r, row, c0)` consumes accumulator columns [c0, c0 + 32) of live output row
// `row`.  `pdl_wait_first`: true waits for the previous kernel on the stream
// before anything reads global memory; false lets the producer and the MMAs start
// at once (X and W are not written by that kernel) and waits in the epilogue.
template <class WLoad, class Epi>
__device__ __forceinline__ void run(const CUtensorMap *tm_x, WLoad wload, int R, int ncols, int dm, Epi epi,
                                    bool pdl_wait_first, int *err, int code0) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
    uint8_t *tiles = smem_raw + pad;
    Smem &sm = *reinterpret_cast<Smem *>(tiles + (size_t)kStages * kStage);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = cluster_ctarank();  // 0 issues the MMAs
    const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
    const int row_blocks = (R + kM - 1) / kM;
    const int col_tiles = (ncols + kN - 1) / kN;
    const int ntiles = row_blocks * col_tiles;
    const int ksteps = (dm + kK - 1) / kK;

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&sm.full[s], 1);   // (even CTA only) its producer, expecting both CTAs' bytes
            mbar_init(&sm.empty[s], 1);  // the even CTA's MMA commit
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&sm.acc_full[a], 1);
            mbar_init(&sm.acc_empty[a], 2);  // (even CTA only) one per epilogue
        }
        mbar_init(&sm.drain, 1);
        sm.abort_flag = 0;
        fence_mbar_init();
    }
    if (pdl_wait_first) asm volatile("griddepcontrol.wait;\n" ::: "memory");
    if (warp == 0) {
        tmem_alloc_pair(&sm.tmem_base, 512);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync();  // both CTAs' barriers initialised and their tensor memory allocated
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;
    volatile int *abort_flag = &sm.abort_flag;
    const uint32_t peer_abort = mapa_shared(&sm.abort_flag, rank ^ 1u);
    auto fail = [&](int code) {
        *abort_flag = 1;
        st_cluster_u32(peer_abort, 1u);
        if (err) atomicExch(err, (int)(kErrMagic | (uint32_t)code));
    };

    if (warp == 0) {
        if (lane == 0) {
            tma_prefetch_desc(tm_x);
            const uint32_t full0 = mapa_shared(&sm.full[0], 0);  // the even CTA's barriers, 8 bytes apart
            uint32_t it = 0;
            bool ok = true;
            for (int tile = pair; tile < ntiles && ok; tile += npairs) {
                const int rb = tile / col_tiles, ct = tile % col_tiles;
                for (int ks = 0; ks < ksteps; ++ks, ++it) {
                    const int s = it % kStages;
                    if (it >= kStages && !(ok = mbar_wait(&sm.empty[s], ((it / kStages) + 1) & 1, abort_flag))) {
                        fail(code0);
                        break;
                    }
                    uint8_t *st = tiles + (size_t)s * kStage;
                    const uint32_t bar = full0 + 8u * (uint32_t)s;
                    if (rank == 0) mbar_arrive_expect_tx(&sm.full[s], 2 * kStage);
                    tma_load_2d_pair(st, tm_x, bar, ks * kK, rb * kM + (int)rank * 128);
#pragma unroll
                    for (int j = 0; j < 2; ++j)
                        wload(st + kAtile + j * (kK * 128), bar, ct * kN + (int)rank * 128 + j * 64, ks * kK);
                }
            }
            // the even CTA waits for the last copies of both CTAs (its barriers count them)
            if (rank == 0) {
                uint32_t first = it > (uint32_t)kStages ? it - kStages : 0;
                for (uint32_t kq = first; kq < it; ++kq)
                    mbar_wait(&sm.full[kq % kStages], (kq / kStages) & 1, abort_flag, 200000000ull);
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {
            const uint32_t idesc = idesc_bf16_f32(kM, kN, false, true);
            uint32_t it = 0, local = 0;
            bool ok = true;
            for (int tile = pair; tile < ntiles && ok; tile += npairs, ++local) {
                const int a = local & 1;
                if (local >= 2 && !(ok = mbar_wait(&sm.acc_empty[a], ((local / 2) + 1) & 1, abort_flag))) {
                    fail(code0 + 1);
                    break;
                }
                tc_fence_after();
                for (int ks = 0; ks < ksteps; ++ks, ++it) {
                    const int s = it % kStages;
                    if (!(ok = mbar_wait(&sm.full[s], (it / kStages) & 1, abort_flag))) {
                        fail(code0 + 2);
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(tiles + (size_t)s * kStage);
                    const uint32_t b_addr = a_addr + kAtile;
#pragma unroll
                    for (int kk = 0; kk < kK / 16; ++kk)
                        mma_ss_pair(tmem + a * kN, smem_desc_sw128(a_addr + kk * 32, 16, 1024),
                                    smem_desc_sw128(b_addr + kk * 2048, kK * 128, 1024), idesc, (ks > 0 || kk > 0));
                    mma_commit_pair(&sm.empty[s], 0x3);
                }
                if (ok) mma_commit_pair(&sm.acc_full[a], 0x3);
            }
            mma_commit_pair(&sm.drain, 0x1);
            mbar_wait(&sm.drain, 0, abort_flag, 200000000ull);
        }
    } else {
        // epilogue: warps 2..5 of each CTA drain that CTA's 128 rows of the tile
        if (!pdl_wait_first) asm volatile("griddepcontrol.wait;\n" ::: "memory");
        const int qq = warp & 3;
        const int rloc = qq * 32 + lane;
        const uint32_t lane_base = (uint32_t)(qq * 32) << 16;
        const uint32_t acc_empty0 = mapa_shared(&sm.acc_empty[0], 0);
        uint32_t local = 0;
        for (int tile = pair; tile < ntiles; tile += npairs, ++local) {
            const int a = local & 1;
            if (rloc == 0) {
                const bool ok = mbar_wait(&sm.acc_full[a], (local / 2) & 1, abort_flag, 4000000000ull);
                if (!ok) fail(code0 + 3);
                sm.go = ok;
            }
            __syncwarp();  // aligned barrier: reconverge the warp first
            asm volatile("bar.sync 1, 128;\n" ::: "memory");
            if (!sm.go) break;
            tc_fence_after();
            const int rb = tile / col_tiles, ct = tile % col_tiles;
            const int row = rb * kM + (int)rank * 128 + rloc;
            const bool live = row < R;
#pragma unroll 1
            for (int cb = 0; cb < kN / 32; ++cb) {
                const int c0 = ct * kN + cb * 32;
                if (c0 >= ncols) break;  // the columns past the matrix (uniform over the CTA)
                uint32_t r[32];
                tmem_ld32(tmem + a * kN + lane_base + cb * 32, r);
                tmem_wait_ld();
                if (live) epi(r, row, c0);
            }
            tc_fence_before();
            __syncwarp();  // aligned barrier: reconverge the warp first
            asm volatile("bar.sync 1, 128;\n" ::: "memory");
            if (rloc == 0) mbar_arrive_cluster(acc_empty0 + 8u * (uint32_t)a);
        }
    }

    // every pair MMA has finished (the even CTA drained them) before either CTA
    // frees its tensor memory or exits with shared memory the peer may still read
    __syncwarp();
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    if (warp == 0) tmem_dealloc_pair(tmem, 512);
}

}  // namespace pairgemm

}  // namespace yoco

namespace yoco_host {

// CTA pairs of `kernel` (cluster of two, pairgemm::kSmemBytes of shared memory)
// that fit the GPU at once; 0 if pairs cannot launch.
inline int pair_gemm_resident_pairs(const void *kernel) {
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)yoco::pairgemm::kSmemBytes) !=
        cudaSuccess)
        return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2);
    cfg.blockDim = dim3(yoco::pairgemm::kThreads);
    cfg.dynamicSmemBytes = yoco::pairgemm::kSmemBytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return n;
}

// Launch configuration of a pair GEMM over `ntiles` 256 x 256 tiles: persistent,
// min(ntiles, resident pairs) pairs, launched as a programmatic dependent of the
// previous kernel on the stream.  `attr` must hold two entries.
inline void pair_gemm_config(cudaLaunchConfig_t &cfg, cudaLaunchAttribute *attr, int ntiles, int pairs,
                             cudaStream_t st) {
    cfg = {};
    cfg.gridDim = dim3(2 * (ntiles < pairs ? ntiles : pairs));
    cfg.blockDim = dim3(yoco::pairgemm::kThreads);
    cfg.dynamicSmemBytes = yoco::pairgemm::kSmemBytes;
    cfg.stream = st;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 2;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
}

}  // namespace yoco_host
