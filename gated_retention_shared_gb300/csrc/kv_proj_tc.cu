// kv_proj_tc.cu -- shared K^/V^ projection on the tensor cores (paper Section 2.2,
// Eq. 2: K^ = RMSNorm(M) W_K, V^ = RMSNorm(M) W_V), bf16, no gain.
//
// out[R, 2n] = M[R, dm] [W_K | W_V] is a plain GEMM; RMSNorm enters as the
// per-row factor r = 1/sqrt(mean(m^2)+eps) (computed by rms_rows_kernel) that
// the epilogue multiplies into the fp32 accumulator before rounding once to
// bf16 and scattering the row into cache slot len + t of its kv heads.
//
// Persistent kernel, one CTA per SM: warp 0 streams 128 x 64 tiles of M and
// 64 x 256 tiles of W into a 4-stage ring with TMA (128-byte swizzle; M K-major,
// W N-major), warp 1 issues tcgen05 MMAs (M=128, N=256, K=16) into one of two
// 256-column TMEM accumulators, warps 2-5 drain the other accumulator.  Tiles
// run row-block major so a block of M is reused from L2 across its 8 column
// tiles and the 12.6 MB of weights stay L2-resident.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"
#include "rope.cuh"
#include "tc.cuh"

namespace yoco {

using namespace tc;

constexpr int kPM = 128, kPN = 256, kPK = 64, kPStages = 4;
constexpr int kPAtile = kPM * kPK * 2;          // 16 KB
constexpr int kPBtile = kPK * kPN * 2;          // 32 KB (4 blocks of 64 columns)
constexpr int kPStage = kPAtile + kPBtile;      // 48 KB
constexpr int kPThreads = 192;

struct ProjSmem {
    uint64_t full[kPStages], empty[kPStages];
    uint64_t acc_full[2], acc_empty[2], drain;
    uint32_t tmem_base;
    int abort_flag;
    int go;  // epilogue continue decision (one writer, read after a barrier)
};

constexpr size_t kPSmem = (size_t)kPStages * kPStage + 1024 + sizeof(ProjSmem);
static_assert(kPSmem <= 232448, "projection tiles and control block must fit shared memory");

__global__ void __launch_bounds__(kPThreads, 1)
proj_tc_kernel(const __grid_constant__ CUtensorMap tm_m, const __grid_constant__ CUtensorMap tm_wk,
               const __grid_constant__ CUtensorMap tm_wv, const float *__restrict__ rrow, bf16_t *__restrict__ kc,
               bf16_t *__restrict__ vc, int R, int T_rows, int dm, int n, int Hkv, int d, int64_t cap, int64_t len,
               int32_t *len_dev, int *err, const float2 *__restrict__ rope_cs) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
    uint8_t *tiles = smem_raw + pad;
    ProjSmem &sm = *reinterpret_cast<ProjSmem *>(tiles + (size_t)kPStages * kPStage);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int row_blocks = (R + kPM - 1) / kPM;
    const int col_tiles = (2 * n) / kPN;
    const int ntiles = row_blocks * col_tiles;
    const int ksteps = (dm + kPK - 1) / kPK;

    if (tid == 0) {
        for (int s = 0; s < kPStages; ++s) {
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
            tma_prefetch_desc(&tm_m);
            tma_prefetch_desc(&tm_wk);
            tma_prefetch_desc(&tm_wv);
            uint32_t it = 0;  // global k-step counter over all tiles of this CTA
            bool ok = true;
            for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
                const int rb = tile / col_tiles, ct = tile % col_tiles;
                const int col0 = ct * kPN;  // within [0, 2n)
                const CUtensorMap *wm = (col0 < n) ? &tm_wk : &tm_wv;
                const int wcol = col0 % n;
                for (int ks = 0; ks < ksteps; ++ks, ++it) {
                    const int s = it % kPStages;
                    if (it >= kPStages && !(ok = mbar_wait(&sm.empty[s], ((it / kPStages) + 1) & 1, abort_flag))) {
                        fail(11);
                        break;
                    }
                    uint8_t *st = tiles + (size_t)s * kPStage;
                    mbar_arrive_expect_tx(&sm.full[s], kPStage);
                    tma_load_2d(st, &tm_m, &sm.full[s], ks * kPK, rb * kPM);
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        tma_load_2d(st + kPAtile + j * (kPK * 128), wm, &sm.full[s], wcol + j * 64, ks * kPK);
                }
            }
            // drain the copies still in flight
            uint32_t first = it > (uint32_t)kPStages ? it - kPStages : 0;
            for (uint32_t k = first; k < it; ++k)
                mbar_wait(&sm.full[k % kPStages], (k / kPStages) & 1, abort_flag, 200000000ull);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16_f32(kPM, kPN, false, true);
            uint32_t it = 0, local = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x, ++local) {
                const int a = local & 1;
                if (local >= 2 && !(ok = mbar_wait(&sm.acc_empty[a], ((local / 2) + 1) & 1, abort_flag))) {
                    fail(12);
                    break;
                }
                tc_fence_after();
                for (int ks = 0; ks < ksteps; ++ks, ++it) {
                    const int s = it % kPStages;
                    if (!(ok = mbar_wait(&sm.full[s], (it / kPStages) & 1, abort_flag))) {
                        fail(13);
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(tiles + (size_t)s * kPStage);
                    const uint32_t b_addr = a_addr + kPAtile;
#pragma unroll
                    for (int kk = 0; kk < kPK / 16; ++kk)
                        mma_ss(tmem + a * kPN, smem_desc_sw128(a_addr + kk * 32, 16, 1024),
                               smem_desc_sw128(b_addr + kk * 2048, kPK * 128, 1024), idesc, (ks > 0 || kk > 0));
                    mma_commit(&sm.empty[s]);
                }
                if (ok) mma_commit(&sm.acc_full[a]);
            }
            // nothing of ours may still run when TMEM is released
            mma_commit(&sm.drain);
            mbar_wait(&sm.drain, 0, abort_flag, 200000000ull);
        }
    } else {
        // epilogue: warps 2..5, TMEM lane quarter = warp % 4.  The RMS factors come
        // from the kernel before this one (a programmatic dependency): wait for it here,
        // while the producer and the MMA warp are already running
        asm volatile("griddepcontrol.wait;\n" ::: "memory");
        const int q = warp & 3;
        const int rloc = q * 32 + lane;

        const uint32_t lane_base = (uint32_t)(q * 32) << 16;
        uint32_t local = 0;
        for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++local) {
            const int a = local & 1;
            if (rloc == 0) {
                const bool ok = mbar_wait(&sm.acc_full[a], (local / 2) & 1, abort_flag, 4000000000ull);
                if (!ok) fail(14);
                sm.go = ok;
            }
            asm volatile("bar.sync 1, 128;\n" ::: "memory");
            if (!sm.go) break;
            tc_fence_after();
            const int rb = tile / col_tiles, ct = tile % col_tiles;
            const int row = rb * kPM + rloc;
            const int col0 = ct * kPN;
            const bool live = row < R;
            const float rs = live ? rrow[row] : 0.f;
            const int bb = live ? row / T_rows : 0, t = live ? row % T_rows : 0;
#pragma unroll 1
            for (int cb = 0; cb < kPN / 32; ++cb) {
                uint32_t r[32];
                tmem_ld32(tmem + a * kPN + lane_base + cb * 32, r);
                tmem_wait_ld();
                if (live) {
                    const int cg = col0 + cb * 32;  // 32 columns inside one head (d is a multiple of 32)
                    bf16_t *dst = (cg < n) ? kc : vc;
                    const int cn = cg % n, h = cn / d, c = cn % d;
                    if (rope_cs && cg < n) {
                        // rotary encoding of K^ at slot position len + t (V is not rotated); the
                        // (cos, sin) table of the call's positions was filled before the GEMM
                        const float2 *cst = rope_cs + (size_t)t * (d / 2) + c / 2;
#pragma unroll
                        for (int e2 = 0; e2 < 16; ++e2) {
                            float x0 = __uint_as_float(r[2 * e2]), x1 = __uint_as_float(r[2 * e2 + 1]);
                            const float2 cs = cst[e2];
                            rope_turn(x0, x1, cs.x, cs.y);
                            r[2 * e2] = __float_as_uint(x0);
                            r[2 * e2 + 1] = __float_as_uint(x1);
                        }
                    }
                    uint4 *p = reinterpret_cast<uint4 *>(dst + (((size_t)bb * Hkv + h) * cap + len + t) * d + c);
#pragma unroll
                    for (int v4 = 0; v4 < 4; ++v4) {
                        uint32_t w[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            __nv_bfloat162 h2 = __floats2bfloat162_rn(__uint_as_float(r[8 * v4 + 2 * e]) * rs,
                                                                       __uint_as_float(r[8 * v4 + 2 * e + 1]) * rs);
                            w[e] = *reinterpret_cast<uint32_t *>(&h2);
                        }
                        p[v4] = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                }
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
    // the last CTA to finish publishes the new length
    if (tid == 0) {
        __threadfence();
        unsigned total = gridDim.x;
        unsigned ticket = atomicAdd(reinterpret_cast<unsigned *>(len_dev + 1), 1u);
        if (ticket == total - 1) {
            len_dev[0] = (int32_t)(len + T_rows);
            __threadfence();
            atomicExch(reinterpret_cast<unsigned *>(len_dev + 1), 0u);
        }
    }
}

}  // namespace yoco

namespace yoco_host {
using namespace yoco;

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        cudaDriverEntryPointQueryResult q;
        void *p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
    }
    return fn;
}

// row-major [rows, cols] bf16, box {64 cols, box_rows rows}, 128-B swizzle
static bool map_2d(CUtensorMap *m, const void *ptr, uint64_t rows, uint64_t cols, uint32_t box_rows) {
    auto enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {64, box_rows};
    cuuint32_t es[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool kv_proj_tc_eligible(const KvProjArgs &a) {
    const int n = a.Hkv * a.d;
    const uintptr_t al = (uintptr_t)a.M | (uintptr_t)a.Wk | (uintptr_t)a.Wv;
    return a.dt == YOCO_BF16 && a.rms_w == nullptr && n % kPN == 0 && a.dm % 8 == 0 && a.dm >= kPK &&
           (int64_t)a.B * a.T >= kPM && (al % 16) == 0;
}

cudaError_t kv_project_append_tc(const KvProjArgs &a, const float *rrow, const float2 *rope_cs, int *err,
                                 cudaStream_t st) {
    const int R = a.B * a.T, n = a.Hkv * a.d;
    CUtensorMap mm, mk, mv;
    if (!map_2d(&mm, a.M, (uint64_t)R, (uint64_t)a.dm, kPM) || !map_2d(&mk, a.Wk, (uint64_t)a.dm, (uint64_t)n, kPK) ||
        !map_2d(&mv, a.Wv, (uint64_t)a.dm, (uint64_t)n, kPK))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(proj_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kPSmem);
    if (e != cudaSuccess) return e;
    const int ntiles = ((R + kPM - 1) / kPM) * (2 * n / kPN);
    const int grid = ntiles < 152 ? ntiles : 152;
    // a programmatic dependent of the RMS pass (M and W are read-only here; the cache
    // slots it writes were last touched by kernels that completed before that pass)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kPThreads);
    cfg.dynamicSmemBytes = kPSmem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    count_launches(1);
    return cudaLaunchKernelEx(&cfg, proj_tc_kernel, mm, mk, mv, rrow, (bf16_t *)a.kc, (bf16_t *)a.vc, R, a.T, a.dm, n,
                              a.Hkv, a.d, a.cap, a.len, a.len_dev, err, rope_cs);
}

}  // namespace yoco_host
