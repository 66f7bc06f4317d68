// kv_proj_tc.cu -- shared K^/V^ projection on the tensor cores (paper Section 2.2,
// Eq. 2: K^ = RMSNorm(M) W_K, V^ = RMSNorm(M) W_V), bf16, no gain.
//
// out[R, 2n] = M[R, dm] [W_K | W_V] is a plain GEMM; RMSNorm enters as the
// per-row factor r = 1/sqrt(mean(m^2)+eps) (computed by rms_rows_kernel) that
// the epilogue multiplies into the fp32 accumulator before rounding once to
// bf16 and scattering the row into cache slot len + t of its kv heads.
//
// The GEMM is the CTA-pair tcgen05 GEMM of pair_gemm.cuh (256 x 256 tiles, 6-stage
// TMA ring, two accumulators in tensor memory); W's columns [0, n) come from W_K
// and [n, 2n) from W_V (n % 256 == 0, so a 64-column block never straddles the
// two).  Tiles run row-block major so a block of M is reused from L2 across its
// column tiles and the 12.6 MB of weights stay L2-resident.  The RMS factors come
// from the kernel before this one (a programmatic dependency, so this grid is
// launched while that pass runs); only the epilogue waits for the pass, but the
// CTAs start as the pass's CTAs leave their SMs, so little runs alongside it.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"
#include "pair_gemm.cuh"
#include "rope.cuh"
#include "tc.cuh"

namespace yoco {

using namespace tc;

__global__ void __launch_bounds__(pairgemm::kThreads, 1)
proj_tc_kernel(const __grid_constant__ CUtensorMap tm_m, const __grid_constant__ CUtensorMap tm_wk,
               const __grid_constant__ CUtensorMap tm_wv, const float *__restrict__ rrow, bf16_t *__restrict__ kc,
               bf16_t *__restrict__ vc, int R, int T_rows, int dm, int n, int Hkv, int d, int64_t cap, int64_t len,
               int32_t *len_dev, int *err, const float2 *__restrict__ rope_cs) {
    auto wload = [&](uint8_t *dst, uint32_t bar, int col, int k0) {
        if (col < n) tma_load_2d_pair(dst, &tm_wk, bar, col, k0);
        else tma_load_2d_pair(dst, &tm_wv, bar, col - n, k0);
    };
    auto epi = [&](uint32_t(&r)[32], int row, int cg) {
        // 32 columns inside one head (d is a multiple of 32) of row `row` = sequence bb, token t
        const float rs = rrow[row];
        const int bb = row / T_rows, t = row % T_rows;
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
        if (!YOCO_DCHECK(len + t < cap && row < R && cg < 2 * n, 0x4B)) return;
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
    };
    pairgemm::run(&tm_m, wload, R, 2 * n, dm, epi, false, err, 11);
    // the last CTA to finish publishes the new length
    if (threadIdx.x == 0) {
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
    return a.dt == YOCO_BF16 && a.rms_w == nullptr && n % pairgemm::kN == 0 && a.dm % 8 == 0 &&
           a.dm >= pairgemm::kK && (int64_t)a.B * a.T >= 128 && (al % 16) == 0;
}

cudaError_t kv_project_append_tc(const KvProjArgs &a, const float *rrow, const float2 *rope_cs, int *err,
                                 cudaStream_t st) {
    static int pairs = -1;
    if (pairs < 0) pairs = pair_gemm_resident_pairs((const void *)proj_tc_kernel);
    if (pairs <= 0) return cudaErrorNotSupported;  // cluster launch unavailable
    const int R = a.B * a.T, n = a.Hkv * a.d;
    CUtensorMap mm, mk, mv;
    if (!map_2d(&mm, a.M, (uint64_t)R, (uint64_t)a.dm, 128) || !map_2d(&mk, a.Wk, (uint64_t)a.dm, (uint64_t)n, 64) ||
        !map_2d(&mv, a.Wv, (uint64_t)a.dm, (uint64_t)n, 64))
        return cudaErrorInvalidValue;
    const int ntiles = ((R + pairgemm::kM - 1) / pairgemm::kM) * (2 * n / pairgemm::kN);
    // a programmatic dependent of the RMS pass (M and W are read-only here; the cache
    // slots it writes were last touched by kernels that completed before that pass)
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    pair_gemm_config(cfg, attr, ntiles, pairs, st);
    // the shared-memory opt-in is set on every launch (it belongs to the current device)
    cudaError_t e = cudaFuncSetAttribute(proj_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)pairgemm::kSmemBytes);
    if (e != cudaSuccess) return e;
    count_launches(1);
    return cudaLaunchKernelEx(&cfg, proj_tc_kernel, mm, mk, mv, rrow, (bf16_t *)a.kc, (bf16_t *)a.vc, R, a.T, a.dm, n,
                              a.Hkv, a.d, a.cap, a.len, a.len_dev, err, rope_cs);
}

}  // namespace yoco_host

YOCO_DEBUG_TU(kv_proj_tc)
