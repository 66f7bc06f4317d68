// attn_fa.cu -- causal softmax attention over a K/V cache for many query rows at
// once (paper Section 2.2, Eq. 3: the cross-decoder's grouped-query attention in
// prefill; with a window it is the sliding-window attention of Section 3.2,
// Eq. 8), bf16, head size 128, on the 5th-generation tensor cores.
//
// One CTA = 128 consecutive query rows of one query head.  Per 128-key tile j:
//     S_j   = Q K_j^T                       (tcgen05, M 128 rows, N 128 keys, TMEM)
//     P_j   = exp(scale S_j - m)  masked    (softmax warps, bf16 written over S_j)
//     O    += P_j V_j                       (tcgen05, A = P_j from TMEM)
// m is a per-row reference maximum that only moves when a tile's maximum passes
// it by more than 8 (natural log units); O is then rescaled in TMEM once.  Every
// P value stays below e^8, the exponent of the final normalisation uses the same
// m, so the result is the plain softmax up to rounding.
//
// Masks: key m is seen by the row at position p when m <= p (causal) and, with
// a window W > 0, p - W < m.  Key tiles outside the block's range are skipped.
//
// Warps: 0 TMA producer (Q once, then K/V tiles through a 3-stage ring), 1 MMA
// issuer (S of tile i is issued before P V of tile i-1, so the softmax of one
// tile overlaps the tensor cores on the other), 2-5 softmax + epilogue (thread =
// TMEM lane = query row).  TMEM: S double buffer at columns 0 / 128, O at 256.
// The GQA group's heads are adjacent in the grid, so their K/V tiles are shared
// through L2.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace yoco {

using namespace tc;

constexpr int kFK = 128;                   // keys per tile = query rows per CTA
constexpr int kFD = 128;                   // head size
constexpr int kFStages = 3;
constexpr int kFTile = kFK * kFD * 2;      // 32 KB bf16 tile
constexpr int kFHalf = kFTile / 2;         // one 64-column block
constexpr int kFThreads = 192;
constexpr uint32_t kColS0 = 0, kColO = 256;
constexpr float kRescaleGap = 8.f;         // m moves only when exceeded by more than this

struct FaSmem {
    uint64_t q_full, full[kFStages], empty[kFStages];
    uint64_t s_full[2], p_ready[2], pv_done[2];
    uint32_t tmem_base;
    int abort_flag;
    int go;
};

constexpr size_t kFTileBytes = (size_t)kFTile + (size_t)kFStages * 2 * kFTile;  // Q + K/V ring
constexpr size_t kFSmem = kFTileBytes + sizeof(FaSmem) + 1024;
static_assert(kFSmem <= 232448, "flash-attention tiles must fit shared memory");

__device__ __forceinline__ void fbar(int n) { asm volatile("bar.sync 1, %0;\n" ::"r"(n) : "memory"); }

__device__ __forceinline__ uint32_t fa_tile_chunk(int r, int c) {  // 16-B chunk c (0..15) of row r, SW128
    return (uint32_t)(c >> 3) * kFHalf + (uint32_t)r * 128u + (uint32_t)(((c & 7) ^ (r & 7)) * 16);
}

__device__ __forceinline__ uint32_t fa_pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h2 = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h2);
}

__global__ void __launch_bounds__(kFThreads, 1)
attn_fa_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o, int T, int Hq,
               int Hkv, int64_t p0, float scale, int64_t window, int *err) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
    uint8_t *tiles = smem_raw + pad;
    uint8_t *sQ = tiles;                      // Q, later the output staging tile
    uint8_t *ring = tiles + kFTile;           // stage s: K at ring + 2 s kFTile, V after it
    FaSmem &sm = *reinterpret_cast<FaSmem *>(tiles + kFTileBytes);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h = blockIdx.x % Hq;
    const int b = blockIdx.x / Hq;
    const int qb = (int)gridDim.y - 1 - (int)blockIdx.y;  // longest rows first
    const int q0 = qb * kFK;
    const int G = Hq / Hkv;
    const int bz = b * Hkv + h / G;  // (sequence, kv head) index of the cache view
    const int64_t pos_lo = p0 + q0;
    const int64_t pos_hi = p0 + min(q0 + kFK, T) - 1;
    const int64_t key_lo = (window > 0) ? max((int64_t)0, pos_lo - window + 1) : 0;
    const int j_lo = (int)(key_lo / kFK), j_hi = (int)(pos_hi / kFK);
    const int ntiles = j_hi - j_lo + 1;

    if (tid == 0) {
        mbar_init(&sm.q_full, 1);
        for (int s = 0; s < kFStages; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&sm.s_full[s], 1);
            mbar_init(&sm.p_ready[s], 1);
            mbar_init(&sm.pv_done[s], 1);
        }
        sm.abort_flag = 0;
        fence_mbar_init();
    }
    // a programmatic dependent of the previous kernel: wait for it before reading Q or the cache
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
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
        // -------------------------------------------------------------- TMA
        if (lane == 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            mbar_arrive_expect_tx(&sm.q_full, kFTile);
            for (int half = 0; half < 2; ++half)
                tma_load_4d(sQ + half * kFHalf, &tm_q, &sm.q_full, half * 64, h, q0, b);
            int i = 0;
            for (; i < ntiles; ++i) {
                const int s = i % kFStages;
                if (i >= kFStages && !mbar_wait(&sm.empty[s], ((i / kFStages) + 1) & 1, abort_flag)) {
                    fail(31);
                    break;
                }
                const int key0 = (j_lo + i) * kFK;
                uint8_t *st = ring + (size_t)s * 2 * kFTile;
                mbar_arrive_expect_tx(&sm.full[s], 2 * kFTile);
                for (int half = 0; half < 2; ++half) {
                    tma_load_3d(st + half * kFHalf, &tm_k, &sm.full[s], half * 64, key0, bz);
                    tma_load_3d(st + kFTile + half * kFHalf, &tm_v, &sm.full[s], half * 64, key0, bz);
                }
            }
            // leave no copy in flight
            mbar_wait(&sm.q_full, 0, abort_flag, 200000000ull);
            for (int k = max(0, i - kFStages); k < i; ++k)
                mbar_wait(&sm.full[k % kFStages], (k / kFStages) & 1, abort_flag, 200000000ull);
        }
    } else if (warp == 1) {
        // -------------------------------------------------------------- MMA
        if (lane == 0) {
            const uint32_t id_s = idesc_bf16_f32(kFK, kFK, false, false);  // A = Q (K-major), B = K (K-major)
            const uint32_t id_o = idesc_bf16_f32(kFK, kFD, false, true);   // A = P (TMEM),   B = V (N-major)
            const uint32_t q_a = smem_u32(sQ);
            bool ok = mbar_wait(&sm.q_full, 0, abort_flag);
            auto issue_pv = [&](int i) -> bool {  // O += P(i) V(i)
                const int s = i % kFStages;
                if (!mbar_wait(&sm.p_ready[i & 1], (i / 2) & 1, abort_flag)) return false;
                tc_fence_after();
                const uint32_t v_a = smem_u32(ring + (size_t)s * 2 * kFTile + kFTile);
                for (int kk = 0; kk < 8; ++kk)
                    mma_ts(tmem + kColO, tmem + kColS0 + 128 * (i & 1) + kk * 8,
                           smem_desc_sw128(v_a + kk * 2048, kFHalf, 1024), id_o, (i > 0 || kk > 0));
                mma_commit(&sm.pv_done[i & 1]);
                mma_commit(&sm.empty[s]);
                return true;
            };
            for (int i = 0; i < ntiles && ok; ++i) {
                const int s = i % kFStages;
                if (!(ok = mbar_wait(&sm.full[s], (i / kFStages) & 1, abort_flag))) break;
                // S buffer i&1 held P(i-2): P V of tile i-2 must be done with it
                if (i >= 2 && !(ok = mbar_wait(&sm.pv_done[i & 1], ((i / 2) - 1) & 1, abort_flag))) break;
                tc_fence_after();
                const uint32_t k_a = smem_u32(ring + (size_t)s * 2 * kFTile);
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t off = (kk >> 2) * kFHalf + (kk & 3) * 32;
                    mma_ss(tmem + kColS0 + 128 * (i & 1), smem_desc_sw128(q_a + off, 16, 1024),
                           smem_desc_sw128(k_a + off, 16, 1024), id_s, kk > 0);
                }
                mma_commit(&sm.s_full[i & 1]);
                if (i > 0 && !(ok = issue_pv(i - 1))) break;
            }
            if (ok && ntiles > 0) ok = issue_pv(ntiles - 1);
            if (!ok) fail(32);
        }
    } else {
        // ------------------------------------------ softmax, rescale, epilogue
        const int q4 = warp & 3;       // TMEM lane quarter of this warp
        const int r = q4 * 32 + lane;  // query row of the block = TMEM lane
        const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
        const int64_t pos = p0 + q0 + r;
        float m_ref = -INFINITY, l = 0.f;
        bool alive = true;
        for (int i = 0; i < ntiles && alive; ++i) {
            if (r == 0) {
                const bool ok = mbar_wait(&sm.s_full[i & 1], (i / 2) & 1, abort_flag);
                if (!ok) fail(33);
                sm.go = ok && !*abort_flag;
            }
            fbar(128);
            if (!sm.go) {
                alive = false;
                break;
            }
            tc_fence_after();
            const uint32_t s_t = tmem + kColS0 + 128 * (i & 1) + lane_base;
            uint32_t sv[128];
#pragma unroll
            for (int cb = 0; cb < 4; ++cb) tmem_ld32(s_t + cb * 32, *reinterpret_cast<uint32_t(*)[32]>(sv + 32 * cb));
            tmem_wait_ld();
            const int64_t key0 = (int64_t)(j_lo + i) * kFK;
            // keys of this tile that row r sees: [lo_c, hi_c)
            const int64_t first = (window > 0) ? pos - window + 1 : 0;
            const int lo_c = (int)max((int64_t)0, min((int64_t)kFK, first - key0));
            const int hi_c = (int)max((int64_t)0, min((int64_t)kFK, pos + 1 - key0));
            float mt = -INFINITY;
#pragma unroll
            for (int c = 0; c < kFK; ++c) {
                const float x = (c >= lo_c && c < hi_c) ? __uint_as_float(sv[c]) * scale : -INFINITY;
                sv[c] = __float_as_uint(x);
                mt = fmaxf(mt, x);
            }
            // move the reference maximum only when this tile passes it by more than the gap
            float alpha = 1.f;
            const bool move = (mt > m_ref + kRescaleGap) || (m_ref == -INFINITY && mt > -INFINITY);
            if (move) {
                alpha = (m_ref == -INFINITY) ? 0.f : __expf(m_ref - mt);
                m_ref = mt;
            }
            // P as packed bf16 over the first 64 columns of S (keys 2c, 2c+1 in column c; every
            // S value is already in registers), 32 keys at a time
            float ls = 0.f;
#pragma unroll
            for (int cb = 0; cb < 4; ++cb) {
                uint32_t pk[16];
#pragma unroll
                for (int c2 = 0; c2 < 16; ++c2) {
                    const float x0 = __uint_as_float(sv[32 * cb + 2 * c2]), x1 = __uint_as_float(sv[32 * cb + 2 * c2 + 1]);
                    const float e0 = (x0 == -INFINITY) ? 0.f : __expf(x0 - m_ref);
                    const float e1 = (x1 == -INFINITY) ? 0.f : __expf(x1 - m_ref);
                    ls += e0 + e1;
                    pk[c2] = fa_pack_bf16x2(e0, e1);
                }
                tmem_st16(s_t + cb * 16, pk);
            }
            l = fmaf(l, alpha, ls);
            tmem_wait_st();
            // O holds tiles < i; a row whose reference moved rescales it before P V of tile i
            // (the whole warp takes part: TMEM loads and stores are warp-wide)
            if (i > 0 && __any_sync(0xffffffffu, move)) {
                bool ok = true;
                if (lane == 0) ok = mbar_wait(&sm.pv_done[(i - 1) & 1], ((i - 1) / 2) & 1, abort_flag);
                ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                if (!ok) {
                    if (lane == 0) fail(34);
                } else {
                    tc_fence_after();
                    const uint32_t o_t = tmem + kColO + lane_base;
#pragma unroll 1
                    for (int cb = 0; cb < 8; ++cb) {
                        uint32_t ov[16];
                        tmem_ld16(o_t + cb * 16, ov);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 16; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
                        tmem_st16(o_t + cb * 16, ov);
                    }
                    tmem_wait_st();
                }
            }
            tc_fence_before();
            fbar(128);  // every row's P (and rescaled O) is in TMEM
            if (r == 0) mbar_arrive(&sm.p_ready[i & 1]);
        }
        // epilogue: o = O / l as bf16, staged in the Q tile (free: every S MMA is done)
        if (alive && ntiles > 0) {
            if (r == 0) {
                const bool ok = mbar_wait(&sm.pv_done[(ntiles - 1) & 1], ((ntiles - 1) / 2) & 1, abort_flag);
                if (!ok) fail(35);
                sm.go = ok && !*abort_flag;
            }
            fbar(128);
            if (sm.go) {
                tc_fence_after();
                const float inv = (l > 0.f) ? 1.f / l : 0.f;
                const uint32_t o_t = tmem + kColO + lane_base;
#pragma unroll 1
                for (int cb = 0; cb < 4; ++cb) {
                    uint32_t ov[32];
                    tmem_ld32(o_t + cb * 32, ov);
                    tmem_wait_ld();
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        *reinterpret_cast<uint4 *>(sQ + fa_tile_chunk(r, cb * 4 + q)) = make_uint4(
                            fa_pack_bf16x2(__uint_as_float(ov[8 * q]) * inv, __uint_as_float(ov[8 * q + 1]) * inv),
                            fa_pack_bf16x2(__uint_as_float(ov[8 * q + 2]) * inv, __uint_as_float(ov[8 * q + 3]) * inv),
                            fa_pack_bf16x2(__uint_as_float(ov[8 * q + 4]) * inv, __uint_as_float(ov[8 * q + 5]) * inv),
                            fa_pack_bf16x2(__uint_as_float(ov[8 * q + 6]) * inv, __uint_as_float(ov[8 * q + 7]) * inv));
                }
                tc_fence_before();
                fence_proxy_async_smem();
                fbar(128);
                if (r == 0) {
                    tma_store_4d(&tm_o, sQ, 0, h, q0, b);  // rows past T are not written
                    tma_store_4d(&tm_o, sQ + kFHalf, 64, h, q0, b);
                    bulk_commit_group();
                    bulk_wait_all();
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

}  // namespace yoco

namespace yoco_host {
using namespace yoco;

static PFN_cuTensorMapEncodeTiled_v12000 fa_encode() {
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

static bool fa_map(CUtensorMap *m, int rank, const void *ptr, const cuuint64_t *dims, const cuuint64_t *strides,
                   const cuuint32_t *box) {
    auto enc = fa_encode();
    if (!enc) return false;
    cuuint32_t es[4] = {1, 1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void *>(ptr), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool attn_fa_eligible(const AttnArgs &a) {
    return a.dt == YOCO_BF16 && a.d == kFD && ((uintptr_t)a.Q % 16) == 0 && ((uintptr_t)a.O % 16) == 0 &&
           a.B <= 65535 && (int64_t)a.B * a.Hq <= 0x7fffffff;
}

cudaError_t attn_fa_launch(const AttnArgs &a, int64_t window, int *err, cudaStream_t st) {
    const int64_t keys = a.p0 + a.T;
    CUtensorMap mq, mk, mv, mo;
    // Q, O: [B, T, Hq, d] as {d, Hq, T, B}, box {64, 1, 128, 1}
    const cuuint64_t qd[4] = {(cuuint64_t)kFD, (cuuint64_t)a.Hq, (cuuint64_t)a.T, (cuuint64_t)a.B};
    const cuuint64_t qs[3] = {(cuuint64_t)kFD * 2, (cuuint64_t)a.Hq * kFD * 2, (cuuint64_t)a.T * a.Hq * kFD * 2};
    const cuuint32_t qbox[4] = {64, 1, (cuuint32_t)kFK, 1};
    // K, V: [B * Hkv, cap, d] viewed with `keys` rows, box {64, 128, 1}
    const cuuint64_t kd[3] = {(cuuint64_t)kFD, (cuuint64_t)keys, (cuuint64_t)a.B * a.Hkv};
    const cuuint64_t ks[2] = {(cuuint64_t)kFD * 2, (cuuint64_t)a.cap * kFD * 2};
    const cuuint32_t kbox[3] = {64, (cuuint32_t)kFK, 1};
    if (!fa_map(&mq, 4, a.Q, qd, qs, qbox) || !fa_map(&mo, 4, a.O, qd, qs, qbox) || !fa_map(&mk, 3, a.kc, kd, ks, kbox) ||
        !fa_map(&mv, 3, a.vc, kd, ks, kbox))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(attn_fa_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kFSmem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(a.B * a.Hq), (unsigned)((a.T + kFK - 1) / kFK));
    cfg.blockDim = dim3(kFThreads);
    cfg.dynamicSmemBytes = kFSmem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    count_launches(1);
    return cudaLaunchKernelEx(&cfg, attn_fa_kernel, mq, mk, mv, mo, a.T, a.Hq, a.Hkv, a.p0, a.scale, window, err);
}

}  // namespace yoco_host
