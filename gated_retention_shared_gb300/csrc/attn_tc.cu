// attn_tc.cu -- cross-decoder attention over the shared K^/V^ cache on the tensor
// cores (paper Section 2.2, Eq. 3: causal grouped-query softmax attention), bf16,
// head size 128, up to 16 query vectors (query rows x heads of one kv group) per CTA.
//
// One CTA = one kv head of one sequence, its group's query vectors and one slice
// of the keys (split-KV; splits are merged by attn_combine_kernel).  Per 128-key
// tile, computed transposed so the short query dimension is the MMA's N:
//     S^T = K Q^T        M = 128 keys,  N = 16 query vectors, K = 128   (TMEM)
//     p   = exp(scale s - m)            one thread per key, online max per vector
//     O^T = V^T P^T      M = 128 dims,  N = 16,                K = 128 keys (TMEM)
//     o   = o * e^{m_old - m_new} + O^T one thread per head dim, fp32 registers
// K and V tiles stream through TMA rings of their own (3 slots each).  A K slot
// is refilled as soon as its S^T MMA completes and a V slot once its O^T MMA
// does, so the next keys' load overlaps the softmax instead of waiting for the
// whole tile to be consumed.  The tensor map's key extent is the number of keys
// the call may read, so slots past it arrive as zeros.  Every
// cross-decoder layer reads the same shared cache, so the loads of each head's
// first keys (half the L2 over all heads) carry normal L2 priority and stay
// cached for the next layer's call, and the rest are marked evict-first.
//
// Warps: 0 TMA producer, 1 MMA issuer, 2-5 softmax + accumulation (thread =
// TMEM lane = key of the tile for S, head dim for O).
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"
#include "rope.cuh"
#include "tc.cuh"

namespace yoco {

using namespace tc;

constexpr int kAK = 128;                      // keys per tile
constexpr int kAD = 128;                      // head size
constexpr int kAN = 16;                       // MMA N: query vectors per CTA (padded)
constexpr int kAStages = 3;
constexpr int kATile = kAK * kAD * 2;         // 32 KB
constexpr int kAHalf = kATile / 2;
constexpr int kAThreads = 192;
constexpr int kAQBytes = kAN * kAD * 2;       // 4 KB: Q (N rows, K-major)
constexpr int kAPBytes = kAN * kAK * 2;       // 4 KB: P^T (N rows of keys, K-major)
constexpr uint32_t kColS = 0, kColOt = 32;    // S^T[2] at 0,16; O^T tiles[2] at 32,48

struct AttnSmem {
    uint64_t full_k[kAStages], full_v[kAStages], empty_k[kAStages], empty_v[kAStages];
    uint64_t s_full[2], s_free[2], p_ready[2], o_full[2], o_free[2], drain;
    uint32_t tmem_base;
    int abort_flag;
    int go;
    float wmax[4][kAN];
    float wsum[4][kAN];
};

constexpr size_t kATileBytes = (size_t)kAStages * 2 * kATile + kAQBytes + 2 * kAPBytes;
constexpr size_t kASmem = kATileBytes + sizeof(AttnSmem) + 1024;
static_assert(kASmem <= 232448, "attention tiles must fit shared memory");

// named barrier 1 (aligned form: the warp is reconverged first, see gret_tc.cu)
__device__ __forceinline__ void abar(int n) {
    __syncwarp();
    asm volatile("bar.sync 1, %0;\n" ::"r"(n) : "memory");
}

// Byte offset of element (row r, col c) in a K-major SW128 tile of `rows` rows
// made of 64-column blocks.
__device__ __forceinline__ uint32_t sw_off(int r, int c, int rows) {
    return (uint32_t)(c >> 6) * rows * 128u + (uint32_t)r * 128u + (uint32_t)((((c & 63) >> 3) ^ (r & 7)) * 16) +
           (uint32_t)(c & 7) * 2u;
}

template <int NQ>
__global__ void __launch_bounds__(kAThreads, 1)
attn_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
               const bf16_t *__restrict__ Q, bf16_t *__restrict__ O, float *__restrict__ part, int T_rows, int Hq,
               int Hkv, int64_t p0, float scale, int RB, int64_t keys_per_split, int splits, int *err,
               float rope_base, const RopeFreq rf, int64_t keep_keys) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
    uint8_t *tiles = smem_raw + pad;
    uint8_t *sQ = tiles + (size_t)kAStages * 2 * kATile;
    uint8_t *sP = sQ + kAQBytes;  // two buffers
    AttnSmem &sm = *reinterpret_cast<AttnSmem *>(sP + 2 * kAPBytes);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = Hq / Hkv;
    const int split = blockIdx.x;
    const int t0 = blockIdx.y * RB;
    const int t1 = min(T_rows, t0 + RB);
    const int bz = blockIdx.z;
    const int b = bz / Hkv, hk = bz % Hkv;
    const int nq = (t1 - t0) * G;
    const int64_t k_lo = (int64_t)split * keys_per_split;
    const int64_t k_hi = min(k_lo + keys_per_split, p0 + (int64_t)t1);
    const int ntiles = (k_hi > k_lo) ? (int)((k_hi - k_lo + kAK - 1) / kAK) : 0;
    (void)YOCO_DCHECK(k_lo >= 0 && t1 <= T_rows && split < splits, 0x50);

    if (tid == 0) {
        for (int s = 0; s < kAStages; ++s) {
            mbar_init(&sm.full_k[s], 1);
            mbar_init(&sm.full_v[s], 1);
            mbar_init(&sm.empty_k[s], 1);
            mbar_init(&sm.empty_v[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&sm.s_full[s], 1);
            mbar_init(&sm.s_free[s], 1);
            mbar_init(&sm.p_ready[s], 1);
            mbar_init(&sm.o_full[s], 1);
            mbar_init(&sm.o_free[s], 1);
        }
        mbar_init(&sm.drain, 1);
        sm.abort_flag = 0;
        fence_mbar_init();
    }
    // The producer (thread 0, which initialised the barriers) starts the first K/V
    // tiles at once, before the programmatic-dependency wait below: the cache is
    // written only by appends, which never release their dependents early, so
    // every append before this call on the stream has completed by the time this
    // grid runs, and the loads overlap the previous kernel's tail.  Q (which the
    // previous kernel may produce) and the workspace (which the previous call's
    // merge may still be reading) are touched only after the wait.
    // L2 priority: the first keep_keys keys of every head stay cached from one call
    // to the next (every cross layer reads this same cache); the rest stream through
    // and are evicted first.
    uint64_t pol_keep = 0, pol_stream = 0;
    int issued = 0;
    // tile i of K (or V) into slot i % kAStages of its ring, whose previous tile is done
    auto issue_tile = [&](int i, bool is_v) {
        const int s = i % kAStages;
        const int key0 = (int)(k_lo + (int64_t)i * kAK);
        uint8_t *dst = tiles + (size_t)s * 2 * kATile + (is_v ? kATile : 0);
        uint64_t *bar = is_v ? &sm.full_v[s] : &sm.full_k[s];
        const uint64_t pol = key0 < keep_keys ? pol_keep : pol_stream;
        mbar_arrive_expect_tx(bar, kATile);
        for (int half = 0; half < 2; ++half)
            tma_load_3d_hint(dst + half * kAHalf, is_v ? &tm_v : &tm_k, bar, half * 64, key0, bz, pol);
    };
    if (tid == 0 && ntiles > 0) {
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        pol_keep = l2_policy_evict_normal();
        pol_stream = l2_policy_evict_first();
        for (; issued < ntiles && issued < kAStages; ++issued) {
            issue_tile(issued, false);
            issue_tile(issued, true);
        }
    }
    // The rest of the prologue that touches nothing of another kernel: both P
    // buffers zero, the TMEM columns, and an L2 prefetch of this CTA's query rows
    // (a prefetch only warms L2, which a later write by the kernel that produces Q
    // updates in place, so the read after the wait still sees that write).
    for (int e = tid; e < 2 * kAPBytes / 16; e += kAThreads) reinterpret_cast<uint4 *>(sP)[e] = make_uint4(0, 0, 0, 0);
    if (tid < 2 * nq) {
        const int n = tid >> 1, t = t0 + n / G, h = hk * G + n % G;
        const bf16_t *row = Q + (((size_t)b * T_rows + t) * Hq + h) * kAD + (tid & 1) * 64;
        asm volatile("prefetch.global.L2 [%0];\n" ::"l"(row));
    }
    if (warp == 0) {
        tmem_alloc(&sm.tmem_base, 64);
        tmem_relinquish();
    }
    // Programmatic dependent launch: the combine grid (and a following call) may
    // start now; apart from the cache tiles and the prefetch above, nothing of
    // another kernel is read or written before the wait, which returns once the
    // previous kernel on the stream has completed (at once when this grid was
    // launched without the attribute).
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
    // Q rows (unscaled bf16) as the K-major B operand; rows >= nq zero
    for (int e = tid; e < kAN * kAD / 8; e += kAThreads) {
        const int n = e / (kAD / 8), c8 = (e % (kAD / 8)) * 8;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (n < nq) {
            const int t = t0 + n / G, h = hk * G + n % G;
            v = *reinterpret_cast<const uint4 *>(Q + (((size_t)b * T_rows + t) * Hq + h) * kAD + c8);
            if (rope_base > 0.f) {  // rotary encoding: turn the row's pairs by its position
                uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    float x0 = __uint_as_float(w[q] << 16), x1 = __uint_as_float(w[q] & 0xFFFF0000u);
                    float c, s;
                    rope_cs_exact(p0 + t, rf.theta[c8 / 2 + q], c, s);
                    rope_turn(x0, x1, c, s);
                    __nv_bfloat162 h2 = __floats2bfloat162_rn(x0, x1);
                    w[q] = *reinterpret_cast<uint32_t *>(&h2);
                }
                v = make_uint4(w[0], w[1], w[2], w[3]);
            }
        }
        *reinterpret_cast<uint4 *>(sQ + sw_off(n, c8, kAN)) = v;
    }
    fence_proxy_async_smem();
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
        if (lane == 0 && ntiles > 0) {
            // The first slots went out before the prologue.  K tile i waits for the
            // S^T MMA of tile i - kAStages, V tile i for its O^T MMA, which the MMA
            // issuer runs after the S^T MMA of the next tile: so K runs ahead.
            volatile int no_abort = 0;
            int i = issued;
            for (; i < ntiles; ++i) {
                const int s = i % kAStages;
                const uint32_t par = ((i / kAStages) + 1) & 1;
                if (i >= kAStages && !mbar_wait(&sm.empty_k[s], par, abort_flag)) {
                    fail(21);
                    break;
                }
                issue_tile(i, false);
                if (i >= kAStages && !mbar_wait(&sm.empty_v[s], par, abort_flag)) {
                    fail(21);
                    mbar_wait(&sm.full_k[s], (i / kAStages) & 1, &no_abort, 200000000ull);
                    break;
                }
                issue_tile(i, true);
            }
            // leave no copy in flight (bounded by time only: an abort must still wait)
            for (int k = max(0, i - kAStages); k < i; ++k) {
                mbar_wait(&sm.full_k[k % kAStages], (k / kAStages) & 1, &no_abort, 200000000ull);
                mbar_wait(&sm.full_v[k % kAStages], (k / kAStages) & 1, &no_abort, 200000000ull);
            }
        }
    } else if (warp == 1) {
        // -------------------------------------------------------------- MMA
        if (lane == 0 && ntiles > 0) {
            const uint32_t id_s = idesc_bf16_f32(kAK, kAN, false, false);  // A = K (K-major), B = Q (K-major)
            const uint32_t id_o = idesc_bf16_f32(kAD, kAN, true, false);   // A = V^T (M-major), B = P^T (K-major)
            const uint32_t q_a = smem_u32(sQ);
            auto issue_s = [&](int i) -> bool {
                const int s = i % kAStages;
                if (!mbar_wait(&sm.full_k[s], (i / kAStages) & 1, abort_flag)) return false;
                if (i >= 2 && !mbar_wait(&sm.s_free[i & 1], ((i / 2) - 1) & 1, abort_flag)) return false;
                tc_fence_after();
                const uint32_t k_a = smem_u32(tiles + (size_t)s * 2 * kATile);
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t off = (kk >> 2) * kAHalf + (kk & 3) * 32;
                    const uint32_t qoff = (kk >> 2) * (kAN * 128) + (kk & 3) * 32;
                    mma_ss(tmem + kColS + 16 * (i & 1), smem_desc_sw128(k_a + off, 16, 1024),
                           smem_desc_sw128(q_a + qoff, 16, 1024), id_s, kk > 0);
                }
                mma_commit(&sm.s_full[i & 1]);
                mma_commit(&sm.empty_k[s]);  // the K slot may be refilled
                return true;
            };
            bool ok = issue_s(0);
            for (int i = 0; i < ntiles && ok; ++i) {
                if (i + 1 < ntiles && !(ok = issue_s(i + 1))) break;
                const int s = i % kAStages;
                if (!(ok = mbar_wait(&sm.p_ready[i & 1], (i / 2) & 1, abort_flag))) break;
                if (i >= 2 && !(ok = mbar_wait(&sm.o_free[i & 1], ((i / 2) - 1) & 1, abort_flag))) break;
                if (!(ok = mbar_wait(&sm.full_v[s], (i / kAStages) & 1, abort_flag))) break;
                tc_fence_after();
                const uint32_t v_a = smem_u32(tiles + (size_t)s * 2 * kATile + kATile);
                const uint32_t p_a = smem_u32(sP + (i & 1) * kAPBytes);
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t poff = (kk >> 2) * (kAN * 128) + (kk & 3) * 32;
                    mma_ss(tmem + kColOt + 16 * (i & 1), smem_desc_sw128(v_a + kk * 2048, kAHalf, 1024),
                           smem_desc_sw128(p_a + poff, 16, 1024), id_o, kk > 0);
                }
                mma_commit(&sm.o_full[i & 1]);
                mma_commit(&sm.empty_v[s]);
            }
            if (!ok) fail(22);
            mma_commit(&sm.drain);
            mbar_wait(&sm.drain, 0, abort_flag, 200000000ull);
        }
    } else {
        // ------------------------------------------ softmax + accumulation
        const int q4 = warp & 3;          // TMEM lane quarter of this warp
        const int r = q4 * 32 + lane;     // key of the tile (S) / head dim (O)
        const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
        float m[NQ], l[NQ], acc[NQ], corr[NQ], corr_prev[NQ];
#pragma unroll
        for (int n = 0; n < NQ; ++n) {
            m[n] = -INFINITY;
            l[n] = 0.f;
            acc[n] = 0.f;
            corr_prev[n] = 1.f;
        }
        auto accumulate = [&](int i) -> bool {  // acc = acc * corr(i) + O^T(i) row r
            if (r == 0) {
                const bool ok = mbar_wait(&sm.o_full[i & 1], (i / 2) & 1, abort_flag);
                if (!ok) fail(23);
                sm.go = ok && !*abort_flag;
            }
            abar(128);
            if (!sm.go) return false;
            tc_fence_after();
            uint32_t o[16];
            tmem_ld16(tmem + kColOt + 16 * (i & 1) + lane_base, o);
            tmem_wait_ld();
#pragma unroll
            for (int n = 0; n < NQ; ++n) acc[n] = fmaf(acc[n], corr_prev[n], __uint_as_float(o[n]));
            tc_fence_before();
            abar(128);
            if (r == 0) mbar_arrive(&sm.o_free[i & 1]);
            return true;
        };
        bool alive = true;
        for (int i = 0; i < ntiles && alive; ++i) {
            if (r == 0) {
                const bool ok = mbar_wait(&sm.s_full[i & 1], (i / 2) & 1, abort_flag);
                if (!ok) fail(24);
                sm.go = ok && !*abort_flag;
            }
            abar(128);
            if (!sm.go) break;
            tc_fence_after();
            uint32_t sv[16];
            tmem_ld16(tmem + kColS + 16 * (i & 1) + lane_base, sv);
            tmem_wait_ld();
            tc_fence_before();
            const int64_t key = k_lo + (int64_t)i * kAK + r;
            float sc[NQ];
            float tmax[NQ];
#pragma unroll
            for (int n = 0; n < NQ; ++n) {
                const int64_t pos = p0 + t0 + n / G;
                const bool ok = n < nq && key < k_hi && key <= pos;
                sc[n] = ok ? scale * __uint_as_float(sv[n]) : -INFINITY;
                float x = sc[n];
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, off));
                tmax[n] = x;
            }
            if (lane == 0) {
#pragma unroll
                for (int n = 0; n < NQ; ++n) sm.wmax[q4][n] = tmax[n];
            }
            abar(128);  // S^T read by everyone; warp maxima visible
            if (r == 0) mbar_arrive(&sm.s_free[i & 1]);
            uint8_t *pb = sP + (i & 1) * kAPBytes;
#pragma unroll
            for (int n = 0; n < NQ; ++n) {
                const float mt = fmaxf(fmaxf(sm.wmax[0][n], sm.wmax[1][n]), fmaxf(sm.wmax[2][n], sm.wmax[3][n]));
                const float mn = fmaxf(m[n], mt);
                corr[n] = (mn == -INFINITY) ? 1.f : __expf(m[n] - mn);
                const float pv = (sc[n] == -INFINITY) ? 0.f : __expf(sc[n] - mn);
                l[n] = fmaf(l[n], corr[n], pv);
                m[n] = mn;
                if (n < nq) {
                    __nv_bfloat16 hb = __float2bfloat16_rn(pv);
                    *reinterpret_cast<__nv_bfloat16 *>(pb + sw_off(n, r, kAN)) = hb;
                }
            }
            fence_proxy_async_smem();
            abar(128);  // P complete; wmax may be rewritten next tile
            if (r == 0) mbar_arrive(&sm.p_ready[i & 1]);
            if (i > 0) alive = accumulate(i - 1);
#pragma unroll
            for (int n = 0; n < NQ; ++n) corr_prev[n] = corr[n];
        }
        if (alive && ntiles > 0) alive = accumulate(ntiles - 1);
        // l: sum of the per-key partial sums over the 128 threads
#pragma unroll
        for (int n = 0; n < NQ; ++n) {
            float x = l[n];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
            if (lane == 0) sm.wsum[q4][n] = x;
        }
        abar(128);
        const int d = r;
#pragma unroll
        for (int n = 0; n < NQ; ++n) {
            if (n >= nq) break;
            const float L = sm.wsum[0][n] + sm.wsum[1][n] + sm.wsum[2][n] + sm.wsum[3][n];
            const int t = t0 + n / G, h = hk * G + n % G;
            const size_t qrow = ((size_t)b * T_rows + t) * Hq + h;
            if (!YOCO_DCHECK(t < T_rows && h < Hq && b < (int)(gridDim.z / Hkv) && split < splits, 0x51)) continue;
            if (splits == 1) {
                O[qrow * kAD + d] = from_f32<bf16_t>(acc[n] / L);
            } else {
                float *pp = part + (qrow * splits + split) * (kAD + 2);
                pp[d] = acc[n];
                if (d == 0) {
                    pp[kAD] = m[n];
                    pp[kAD + 1] = L;
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 64);
}

}  // namespace yoco

namespace yoco_host {
using namespace yoco;

static PFN_cuTensorMapEncodeTiled_v12000 attn_encode() {
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

// cache [B*Hkv, cap, 128] bf16 viewed with `keys` rows per (b, kv head)
static bool cache_map(CUtensorMap *m, const void *ptr, int64_t bhk, int64_t cap, int64_t keys) {
    auto enc = attn_encode();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)kAD, (cuuint64_t)keys, (cuuint64_t)bhk};
    cuuint64_t strides[2] = {(cuuint64_t)kAD * 2, (cuuint64_t)cap * kAD * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)kAK, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Bytes of the shared cache that decode calls keep in L2 between calls: half of
// the L2 (about 64 MB on GB300).  Measured on a 134 MB cache read by back-to-back
// calls: keeping 64 MB takes a call from 29.7 to 24.4-24.9 us; keeping 96 MB or
// more gives the time back, as lines start to evict each other.
static int64_t attn_l2_keep_bytes() {
    static int64_t bytes = -1;
    if (bytes < 0) {
        int dev = 0, l2 = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev) != cudaSuccess)
            l2 = 0;
        bytes = (int64_t)l2 / 2;
    }
    return bytes;
}

bool attn_tc_eligible(const AttnArgs &a, int nq) {
    return a.dt == YOCO_BF16 && a.d == kAD && nq <= kAN && ((uintptr_t)a.Q % 16) == 0;
}

cudaError_t attn_tc_launch(const AttnArgs &a, int RB, int nq, int64_t kps, int splits, void *ws, int *err,
                           cudaStream_t st) {
    const int64_t keys = a.p0 + a.T;
    CUtensorMap mk, mv;
    if (!cache_map(&mk, a.kc, (int64_t)a.B * a.Hkv, a.cap, keys) || !cache_map(&mv, a.vc, (int64_t)a.B * a.Hkv, a.cap, keys))
        return cudaErrorInvalidValue;
    dim3 grid(splits, (a.T + RB - 1) / RB, a.B * a.Hkv);
    const RopeFreq rf = make_rope_freq(a.rope_base, kAD);
    const int64_t keep_keys = attn_l2_keep_bytes() / ((int64_t)a.B * a.Hkv * kAD * 2 * 2);
    cudaError_t e;
    // launched as a programmatic dependent of the previous kernel on the stream: its
    // prologue (barriers, TMEM, descriptor prefetch) overlaps that kernel's tail
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kAThreads);
    cfg.dynamicSmemBytes = kASmem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
#define YOCO_ATTN_TC(NQ_)                                                                                          \
    e = cudaFuncSetAttribute(attn_tc_kernel<NQ_>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kASmem);       \
    if (e != cudaSuccess) return e;                                                                                \
    e = cudaLaunchKernelEx(&cfg, attn_tc_kernel<NQ_>, mk, mv, (const bf16_t *)a.Q, (bf16_t *)a.O, (float *)ws,     \
                           a.T, a.Hq, a.Hkv, a.p0, a.scale, RB, kps, splits, err, a.rope_base, rf, keep_keys);               \
    if (e != cudaSuccess) return e;
    if (nq <= 4) {
        YOCO_ATTN_TC(4)
    } else if (nq <= 8) {
        YOCO_ATTN_TC(8)
    } else {
        YOCO_ATTN_TC(16)
    }
#undef YOCO_ATTN_TC
    return cudaGetLastError();
}

}  // namespace yoco_host

YOCO_DEBUG_TU(attn_tc)
