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
// The GEMM is the CTA-pair tcgen05 GEMM of pair_gemm.cuh (256 x 256 tiles, the
// even CTA issuing 256 x 256 x 16 MMAs over both CTAs' halves); this file adds
// the epilogue.  W's last column tile is partly past the matrix and arrives
// zero-filled.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"
#include "pair_gemm.cuh"
#include "tc.cuh"

namespace yoco {

using namespace tc;

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

__global__ void __launch_bounds__(pairgemm::kThreads, 1)
qkvg_tc_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w, int R, int N, int dm,
               int H, int d, bf16_t *__restrict__ q, bf16_t *__restrict__ k, bf16_t *__restrict__ v,
               float *__restrict__ logits, const float2 *__restrict__ rope_cs, int *err) {
    auto wload = [&](uint8_t *dst, uint32_t bar, int col, int k0) { tma_load_2d_pair(dst, &tm_w, bar, col, k0); };
    // row = b N + t: position t inside its sequence for the rotary table
    auto epi = [&](uint32_t(&r)[32], int row, int c0) {
        qkvg_store32(r, row, row % N, c0, H, d, q, k, v, logits, rope_cs);
    };
    // a programmatic dependent of the previous kernel: wait for it before reading X or W
    pairgemm::run(&tm_x, wload, R, 3 * H * d + H, dm, epi, true, err, 41);
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

cudaError_t qkvg_project(const void *X, const void *W, int B, int N, int dm, int H, int d, void *q, void *k, void *v,
                         float *logits, const float2 *rope_cs, int *err, cudaStream_t st) {
    static int pairs = -1;
    if (pairs < 0) pairs = pair_gemm_resident_pairs((const void *)qkvg_tc_kernel);
    if (pairs <= 0) return cudaErrorNotSupported;  // cluster launch unavailable
    const int R = B * N;
    const int ncols = 3 * H * d + H;
    CUtensorMap mx, mw;
    if (!qkvg_map(&mx, X, (uint64_t)R, (uint64_t)dm, 128) || !qkvg_map(&mw, W, (uint64_t)dm, (uint64_t)ncols, 64))
        return cudaErrorInvalidValue;
    const int ntiles = ((R + pairgemm::kM - 1) / pairgemm::kM) * ((ncols + pairgemm::kN - 1) / pairgemm::kN);
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    pair_gemm_config(cfg, attr, ntiles, pairs, st);
    // the shared-memory opt-in is set on every launch (it belongs to the current device)
    cudaError_t e = cudaFuncSetAttribute(qkvg_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)pairgemm::kSmemBytes);
    if (e != cudaSuccess) return e;
    count_launches(1);
    return cudaLaunchKernelEx(&cfg, qkvg_tc_kernel, mx, mw, R, N, dm, H, d, (bf16_t *)q, (bf16_t *)k, (bf16_t *)v,
                              logits, rope_cs, err);
}

}  // namespace yoco_host

YOCO_DEBUG_TU(qkvg_tc)
