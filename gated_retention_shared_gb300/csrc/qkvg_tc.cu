// qkvg_tc.cu -- the gated-retention layer's input projections in one GEMM on the
// tensor cores (paper Section 3.1: Q = (X W_Q) (.) Theta, K = (X W_K) (.) conj(Theta),
// V = X W_V, gamma = sigmoid(X W_gamma)^(1/tau)), bf16 in, fp32 accumulate.
//
//     [q | k | v | logits] = X [W_Q | W_K | W_V | W_gamma]      X [R, dm], W [dm, 3 H d + H]
//
// X is read once for all four projections.  The epilogue writes q, k, v straight
// into the token-major [B, N, H, d] layout the chunkwise kernel reads (turning q
// and k by their positions when rotary encoding is on, from a per-call cos/sin
// table) and the gate logits as fp32 [B, N, H]; the chunk kernel's decay scan
// applies logsigmoid / tau as it reads them.
//
// Persistent kernel, one CTA per SM, the same shape as the shared-K/V projection:
// warp 0 streams 128 x 64 tiles of X and 64 x 256 tiles of W (4-stage TMA ring,
// 128-byte swizzle; W's last column tile is partly past the matrix and arrives
// zero-filled), warp 1 issues tcgen05 MMAs into one of two 256-column TMEM
// accumulators, warps 2-5 drain the other.  Row-block-major tile order keeps a
// block of X in L2 across its column tiles.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace yoco {

using namespace tc;

constexpr int kGM = 128, kGN = 256, kGK = 64, kGStages = 4;
constexpr int kGAtile = kGM * kGK * 2;          // 16 KB
constexpr int kGBtile = kGK * kGN * 2;          // 32 KB (4 blocks of 64 columns)
constexpr int kGStage = kGAtile + kGBtile;      // 48 KB
constexpr int kGThreads = 192;

struct QkvgSmem {
    uint64_t full[kGStages], empty[kGStages];
    uint64_t acc_full[2], acc_empty[2], drain;
    uint32_t tmem_base;
    int abort_flag;
    int go;
};

constexpr size_t kGSmem = (size_t)kGStages * kGStage + 1024 + sizeof(QkvgSmem);
static_assert(kGSmem <= 232448, "projection tiles and control block must fit shared memory");

// Write 32 accumulator columns [c0, c0 + 32) of output row `row` (position t in its
// sequence): into q, k or v (turned by the rotary table when it is given) or, past
// 3 H d, into the gate logits.
__device__ __forceinline__ void qkvg_store32(uint32_t (&r)[32], int row, int t, int c0, int H, int d,
                                             bf16_t *__restrict__ q, bf16_t *__restrict__ k, bf16_t *__restrict__ v,
                                             float *__restrict__ logits, const float2 *__restrict__ rope_cs) {
    const int Hd = H * d;
    if (c0 < 3 * Hd) {
        // q, k or v: 32 columns inside one head (d is a multiple of 32)
        const int region = c0 / Hd, within = c0 % Hd;
        bf16_t *dst = (region == 0 ? q : region == 1 ? k : v) + (size_t)row * Hd + within;
        if (rope_cs && region < 2) {  // rotary encoding of q and k at position pos0 + t
            const float2 *cst = rope_cs + (size_t)t * (d / 2) + (within % d) / 2;
#pragma unroll
            for (int e2 = 0; e2 < 16; ++e2) {
                const float2 cs = cst[e2];
                const float x0 = __uint_as_float(r[2 * e2]), x1 = __uint_as_float(r[2 * e2 + 1]);
                r[2 * e2] = __float_as_uint(x0 * cs.x - x1 * cs.y);
                r[2 * e2 + 1] = __float_as_uint(x0 * cs.y + x1 * cs.x);
            }
        }
        uint4 *p = reinterpret_cast<uint4 *>(dst);
#pragma unroll
        for (int v4 = 0; v4 < 4; ++v4) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                __nv_bfloat162 h2 =
                    __floats2bfloat162_rn(__uint_as_float(r[8 * v4 + 2 * e]), __uint_as_float(r[8 * v4 + 2 * e + 1]));
                w[e] = *reinterpret_cast<uint32_t *>(&h2);
            }
            p[v4] = make_uint4(w[0], w[1], w[2], w[3]);
        }
    } else {
        // gate logits x . w_gamma, one per head
        const int g0 = c0 - 3 * Hd;
#pragma unroll
        for (int e = 0; e < 32; ++e)
            if (g0 + e < H) logits[(size_t)row * H + g0 + e] = __uint_as_float(r[e]);
    }
}

__global__ void __launch_bounds__(kGThreads, 1)
qkvg_tc_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w, int R, int N, int dm,
               int H, int d, bf16_t *__restrict__ q, bf16_t *__restrict__ k, bf16_t *__restrict__ v,
               float *__restrict__ logits, const float2 *__restrict__ rope_cs, int *err) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
    uint8_t *tiles = smem_raw + pad;
    QkvgSmem &sm = *reinterpret_cast<QkvgSmem *>(tiles + (size_t)kGStages * kGStage);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int Hd = H * d;
    const int ncols = 3 * Hd + H;
    const int row_blocks = (R + kGM - 1) / kGM;
    const int col_tiles = (ncols + kGN - 1) / kGN;
    const int ntiles = row_blocks * col_tiles;
    const int ksteps = (dm + kGK - 1) / kGK;

    if (tid == 0) {
        for (int s = 0; s < kGStages; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&sm.acc_full[a], 1);
            mbar_init(&sm.acc_empty[a], 1);
        }
        mbar_init(&sm.drain, 1);
        sm.abort_flag = 0;
        fence_mbar_init();
    }
    // a programmatic dependent of the previous kernel: wait for it before reading X or W
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
    if (warp == 0) {
        tmem_alloc(&sm.tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;
    volatile int *abort_flag = &sm.abort_flag;
    auto fail = [&](int code) {
        *abort_flag = 1;
        if (err) atomicExch(err, (int)(kErrMagic | (uint32_t)code));
    };

    if (warp == 0) {
        if (lane == 0) {
            tma_prefetch_desc(&tm_x);
            tma_prefetch_desc(&tm_w);
            uint32_t it = 0;  // global k-step counter over all tiles of this CTA
            bool ok = true;
            for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
                const int rb = tile / col_tiles, ct = tile % col_tiles;
                for (int ks = 0; ks < ksteps; ++ks, ++it) {
                    const int s = it % kGStages;
                    if (it >= kGStages && !(ok = mbar_wait(&sm.empty[s], ((it / kGStages) + 1) & 1, abort_flag))) {
                        fail(41);
                        break;
                    }
                    uint8_t *st = tiles + (size_t)s * kGStage;
                    mbar_arrive_expect_tx(&sm.full[s], kGStage);
                    tma_load_2d(st, &tm_x, &sm.full[s], ks * kGK, rb * kGM);
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        tma_load_2d(st + kGAtile + j * (kGK * 128), &tm_w, &sm.full[s], ct * kGN + j * 64, ks * kGK);
                }
            }
            // drain the copies still in flight
            uint32_t first = it > (uint32_t)kGStages ? it - kGStages : 0;
            for (uint32_t kq = first; kq < it; ++kq)
                mbar_wait(&sm.full[kq % kGStages], (kq / kGStages) & 1, abort_flag, 200000000ull);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16_f32(kGM, kGN, false, true);
            uint32_t it = 0, local = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x, ++local) {
                const int a = local & 1;
                if (local >= 2 && !(ok = mbar_wait(&sm.acc_empty[a], ((local / 2) + 1) & 1, abort_flag))) {
                    fail(42);
                    break;
                }
                tc_fence_after();
                for (int ks = 0; ks < ksteps; ++ks, ++it) {
                    const int s = it % kGStages;
                    if (!(ok = mbar_wait(&sm.full[s], (it / kGStages) & 1, abort_flag))) {
                        fail(43);
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(tiles + (size_t)s * kGStage);
                    const uint32_t b_addr = a_addr + kGAtile;
#pragma unroll
                    for (int kk = 0; kk < kGK / 16; ++kk)
                        mma_ss(tmem + a * kGN, smem_desc_sw128(a_addr + kk * 32, 16, 1024),
                               smem_desc_sw128(b_addr + kk * 2048, kGK * 128, 1024), idesc, (ks > 0 || kk > 0));
                    mma_commit(&sm.empty[s]);
                }
                if (ok) mma_commit(&sm.acc_full[a]);
            }
            mma_commit(&sm.drain);
            mbar_wait(&sm.drain, 0, abort_flag, 200000000ull);
        }
    } else {
        // epilogue: warps 2..5, TMEM lane quarter = warp % 4, thread = output row
        const int qq = warp & 3;
        const int rloc = qq * 32 + lane;
        const uint32_t lane_base = (uint32_t)(qq * 32) << 16;
        uint32_t local = 0;
        for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++local) {
            const int a = local & 1;
            if (rloc == 0) {
                const bool ok = mbar_wait(&sm.acc_full[a], (local / 2) & 1, abort_flag, 4000000000ull);
                if (!ok) fail(44);
                sm.go = ok;
            }
            asm volatile("bar.sync 1, 128;\n" ::: "memory");
            if (!sm.go) break;
            tc_fence_after();
            const int rb = tile / col_tiles, ct = tile % col_tiles;
            const int row = rb * kGM + rloc;
            const bool live = row < R;
            const int t = live ? row % N : 0;  // position of the row inside its sequence
#pragma unroll 1
            for (int cb = 0; cb < kGN / 32; ++cb) {
                const int c0 = ct * kGN + cb * 32;  // first of these 32 columns of [W_Q | W_K | W_V | W_gamma]
                if (c0 >= ncols) break;             // the columns past the matrix (uniform over the CTA)
                uint32_t r[32];
                tmem_ld32(tmem + a * kGN + lane_base + cb * 32, r);
                tmem_wait_ld();
                if (live) qkvg_store32(r, row, t, c0, H, d, q, k, v, logits, rope_cs);
            }
            tc_fence_before();
            // all four epilogue warps must be done with this accumulator
            asm volatile("bar.sync 1, 128;\n" ::: "memory");
            if (rloc == 0) mbar_arrive(&sm.acc_empty[a]);
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

// ------------------------------------------------------------------ CTA pairs
// The same product on 256 x 256 tiles computed by a pair of CTAs (a cluster of
// two) with one tcgen05 MMA of shape 256 x 256 x 16 issued by the even CTA: each
// CTA stages its own 128 rows of X and its own 128 of the 256 W columns, and the
// MMA reads the other half from the peer's shared memory.  Against the one-CTA
// tile this halves the W bytes every SM stages and reads per MMA (32 KB per
// 64-deep step instead of 48 KB for the same work per SM).
//   * both CTAs' copies of a stage complete on the even CTA's `full` barrier,
//     whose one arrival (the even producer's) expects the 64 KB of both; a peer
//     copy that lands before that arrival leaves the phase pending, and the odd
//     producer refills a stage only after the MMA freed it, i.e. after the phase;
//   * the even CTA's MMA commit frees the stage in both CTAs (`empty`, multicast)
//     and announces a finished accumulator to both epilogues (`acc_full`);
//   * both epilogues hand the accumulator back on the even CTA's `acc_empty`.
constexpr int kPM = 256, kPStages = 6;
constexpr int kPAtile = 128 * kGK * 2;         // 16 KB: this CTA's 128 rows of X
constexpr int kPBtile = kGK * 128 * 2;         // 16 KB: this CTA's 128 columns of W
constexpr int kPStage = kPAtile + kPBtile;     // 32 KB

struct QkvgPairSmem {
    uint64_t full[kPStages], empty[kPStages];
    uint64_t acc_full[2], acc_empty[2], drain;
    uint32_t tmem_base;
    int abort_flag;
    int go;
};

constexpr size_t kPSmemBytes = (size_t)kPStages * kPStage + 1024 + sizeof(QkvgPairSmem);
static_assert(kPSmemBytes <= 232448, "pair tiles and control block must fit shared memory");

__global__ void __launch_bounds__(kGThreads, 1)
qkvg_tc_pair_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w, int R,
                    int N, int dm, int H, int d, bf16_t *__restrict__ q, bf16_t *__restrict__ k,
                    bf16_t *__restrict__ v, float *__restrict__ logits, const float2 *__restrict__ rope_cs, int *err) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
    uint8_t *tiles = smem_raw + pad;
    QkvgPairSmem &sm = *reinterpret_cast<QkvgPairSmem *>(tiles + (size_t)kPStages * kPStage);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = cluster_ctarank();  // 0 issues the MMAs
    const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
    const int ncols = 3 * H * d + H;
    const int row_blocks = (R + kPM - 1) / kPM;
    const int col_tiles = (ncols + kGN - 1) / kGN;
    const int ntiles = row_blocks * col_tiles;
    const int ksteps = (dm + kGK - 1) / kGK;

    if (tid == 0) {
        for (int s = 0; s < kPStages; ++s) {
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
    // a programmatic dependent of the previous kernel: wait for it before reading X or W
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
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
            tma_prefetch_desc(&tm_x);
            tma_prefetch_desc(&tm_w);
            const uint32_t full0 = mapa_shared(&sm.full[0], 0);  // the even CTA's barriers, 8 bytes apart
            uint32_t it = 0;
            bool ok = true;
            for (int tile = pair; tile < ntiles && ok; tile += npairs) {
                const int rb = tile / col_tiles, ct = tile % col_tiles;
                for (int ks = 0; ks < ksteps; ++ks, ++it) {
                    const int s = it % kPStages;
                    if (it >= kPStages && !(ok = mbar_wait(&sm.empty[s], ((it / kPStages) + 1) & 1, abort_flag))) {
                        fail(45);
                        break;
                    }
                    uint8_t *st = tiles + (size_t)s * kPStage;
                    const uint32_t bar = full0 + 8u * (uint32_t)s;
                    if (rank == 0) mbar_arrive_expect_tx(&sm.full[s], 2 * kPStage);
                    tma_load_2d_pair(st, &tm_x, bar, ks * kGK, rb * kPM + (int)rank * 128);
#pragma unroll
                    for (int j = 0; j < 2; ++j)
                        tma_load_2d_pair(st + kPAtile + j * (kGK * 128), &tm_w, bar,
                                         ct * kGN + (int)rank * 128 + j * 64, ks * kGK);
                }
            }
            // the even CTA waits for the last copies of both CTAs (its barriers count them)
            if (rank == 0) {
                uint32_t first = it > (uint32_t)kPStages ? it - kPStages : 0;
                for (uint32_t kq = first; kq < it; ++kq)
                    mbar_wait(&sm.full[kq % kPStages], (kq / kPStages) & 1, abort_flag, 200000000ull);
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {
            const uint32_t idesc = idesc_bf16_f32(kPM, kGN, false, true);
            uint32_t it = 0, local = 0;
            bool ok = true;
            for (int tile = pair; tile < ntiles && ok; tile += npairs, ++local) {
                const int a = local & 1;
                if (local >= 2 && !(ok = mbar_wait(&sm.acc_empty[a], ((local / 2) + 1) & 1, abort_flag))) {
                    fail(46);
                    break;
                }
                tc_fence_after();
                for (int ks = 0; ks < ksteps; ++ks, ++it) {
                    const int s = it % kPStages;
                    if (!(ok = mbar_wait(&sm.full[s], (it / kPStages) & 1, abort_flag))) {
                        fail(47);
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(tiles + (size_t)s * kPStage);
                    const uint32_t b_addr = a_addr + kPAtile;
#pragma unroll
                    for (int kk = 0; kk < kGK / 16; ++kk)
                        mma_ss_pair(tmem + a * kGN, smem_desc_sw128(a_addr + kk * 32, 16, 1024),
                                    smem_desc_sw128(b_addr + kk * 2048, kGK * 128, 1024), idesc, (ks > 0 || kk > 0));
                    mma_commit_pair(&sm.empty[s], 0x3);
                }
                if (ok) mma_commit_pair(&sm.acc_full[a], 0x3);
            }
            mma_commit_pair(&sm.drain, 0x1);
            mbar_wait(&sm.drain, 0, abort_flag, 200000000ull);
        }
    } else {
        // epilogue: warps 2..5 of each CTA drain that CTA's 128 rows of the tile
        const int qq = warp & 3;
        const int rloc = qq * 32 + lane;
        const uint32_t lane_base = (uint32_t)(qq * 32) << 16;
        const uint32_t acc_empty0 = mapa_shared(&sm.acc_empty[0], 0);
        uint32_t local = 0;
        for (int tile = pair; tile < ntiles; tile += npairs, ++local) {
            const int a = local & 1;
            if (rloc == 0) {
                const bool ok = mbar_wait(&sm.acc_full[a], (local / 2) & 1, abort_flag, 4000000000ull);
                if (!ok) fail(48);
                sm.go = ok;
            }
            asm volatile("bar.sync 1, 128;\n" ::: "memory");
            if (!sm.go) break;
            tc_fence_after();
            const int rb = tile / col_tiles, ct = tile % col_tiles;
            const int row = rb * kPM + (int)rank * 128 + rloc;
            const bool live = row < R;
            const int t = live ? row % N : 0;
#pragma unroll 1
            for (int cb = 0; cb < kGN / 32; ++cb) {
                const int c0 = ct * kGN + cb * 32;
                if (c0 >= ncols) break;
                uint32_t r[32];
                tmem_ld32(tmem + a * kGN + lane_base + cb * 32, r);
                tmem_wait_ld();
                if (live) qkvg_store32(r, row, t, c0, H, d, q, k, v, logits, rope_cs);
            }
            tc_fence_before();
            asm volatile("bar.sync 1, 128;\n" ::: "memory");
            if (rloc == 0) mbar_arrive_cluster(acc_empty0 + 8u * (uint32_t)a);
        }
    }

    // every pair MMA has finished (the even CTA drained them) before either CTA
    // frees its tensor memory or exits with shared memory the peer may still read
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    if (warp == 0) tmem_dealloc_pair(tmem, 512);
}

}  // namespace yoco

namespace yoco_host {
using namespace yoco;

static PFN_cuTensorMapEncodeTiled_v12000 qkvg_encode() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        cudaDriverEntryPointQueryResult qr;
        void *p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &qr) ==
                cudaSuccess &&
            qr == cudaDriverEntryPointSuccess)
            fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
    }
    return fn;
}

// row-major [rows, cols] bf16, box {64 cols, box_rows rows}, 128-B swizzle
static bool qkvg_map(CUtensorMap *m, const void *ptr, uint64_t rows, uint64_t cols, uint32_t box_rows) {
    auto enc = qkvg_encode();
    if (!enc) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {64, box_rows};
    cuuint32_t es[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// CTA pairs that fit the GPU at once (one CTA per SM); 0 if pairs cannot launch
static int qkvg_pairs_resident() {
    static int pairs = -1;
    if (pairs < 0) {
        pairs = 0;
        if (cudaFuncSetAttribute(qkvg_tc_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kPSmemBytes) != cudaSuccess)
            return pairs;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2);
        cfg.blockDim = dim3(kGThreads);
        cfg.dynamicSmemBytes = kPSmemBytes;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, qkvg_tc_pair_kernel, &cfg) == cudaSuccess) pairs = n;
        else (void)cudaGetLastError();
    }
    return pairs;
}

cudaError_t qkvg_project(const void *X, const void *W, int B, int N, int dm, int H, int d, void *q, void *k, void *v,
                         float *logits, const float2 *rope_cs, int *err, cudaStream_t st) {
    const int R = B * N;
    const int ncols = 3 * H * d + H;
    const int col_tiles = (ncols + kGN - 1) / kGN;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kGThreads);
    cfg.stream = st;
    cfg.attrs = attr;
    CUtensorMap mx, mw;
    const int pairs = qkvg_pairs_resident();
    if (pairs > 0) {
        if (!qkvg_map(&mx, X, (uint64_t)R, (uint64_t)dm, 128) || !qkvg_map(&mw, W, (uint64_t)dm, (uint64_t)ncols, kGK))
            return cudaErrorInvalidValue;
        const int ntiles = ((R + kPM - 1) / kPM) * col_tiles;
        cfg.gridDim = dim3(2 * (ntiles < pairs ? ntiles : pairs));
        cfg.dynamicSmemBytes = kPSmemBytes;
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = 2;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
        count_launches(1);
        return cudaLaunchKernelEx(&cfg, qkvg_tc_pair_kernel, mx, mw, R, N, dm, H, d, (bf16_t *)q, (bf16_t *)k,
                                  (bf16_t *)v, logits, rope_cs, err);
    }
    if (!qkvg_map(&mx, X, (uint64_t)R, (uint64_t)dm, kGM) || !qkvg_map(&mw, W, (uint64_t)dm, (uint64_t)ncols, kGK))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(qkvg_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGSmem);
    if (e != cudaSuccess) return e;
    const int ntiles = ((R + kGM - 1) / kGM) * col_tiles;
    cfg.gridDim = dim3(ntiles < 152 ? ntiles : 152);
    cfg.dynamicSmemBytes = kGSmem;
    cfg.numAttrs = 1;
    count_launches(1);
    return cudaLaunchKernelEx(&cfg, qkvg_tc_kernel, mx, mw, R, N, dm, H, d, (bf16_t *)q, (bf16_t *)k, (bf16_t *)v,
                              logits, rope_cs, err);
}

}  // namespace yoco_host
