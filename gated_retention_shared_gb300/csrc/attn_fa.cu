// attn_fa.cu -- causal softmax attention over a K/V cache for many query rows at
// once (paper Section 2.2, Eq. 3: the cross-decoder's grouped-query attention in
// prefill; with a window it is the sliding-window attention of Section 3.2,
// Eq. 8), bf16, head size 128, on the 5th-generation tensor cores.
//
// One CTA = 256 consecutive query rows of one query head, as two sets of 128
// (A: rows 0..127, B: rows 128..255), each with its own softmax warpgroup, so the
// tensor cores work on one set while the other set's softmax runs.  Per 128-key
// tile j and set X:
//     S_X   = Q_X K_j^T                     (tcgen05, M 128 rows, N 128 keys, TMEM)
//     P_X   = 2^(c S_X - m)  masked         (softmax warps, bf16 into shared memory)
//     O_X  += P_X V_j                       (tcgen05, A = P_X from shared memory)
// with c = scale * log2(e) and m a per-row reference maximum (base-2 units) that
// only moves when a tile's maximum passes it by more than 8 / ln 2 (so by e^8);
// O_X is then rescaled in TMEM once.  Every P value stays below e^8 and the final
// normalisation uses the same m, so the result is the plain softmax up to rounding.
//
// Masks: key m is seen by the row at position p when m <= p (causal) and, with
// a window W > 0, p - W < m.  Only tiles that cross a row's boundary are masked
// element by element; key tiles outside the CTA's range are skipped.
//
// Warps: 0 TMA producer (Q_A, Q_B once, then K and V tiles through 2-stage rings
// with barriers of their own), 1 MMA issuer, 2-5 softmax + epilogue of set A, 6-9
// of set B (thread = TMEM lane = query row).  A set's softmax warps read S_X(j)
// out of TMEM and free it at once, so S_X(j + 1) is computed while they work;
// the two sets write P in turn into one shared-memory buffer (B's P(j) after
// P_A V(j), A's P(j + 1) after P_B V(j)), each 64-key half as soon as the other
// set's MMAs have read that half.  Tensor-core order per tile:
// S_A(j + 1), P_A V(j), S_B(j + 1), P_B V(j): each S sits between the P V MMAs.
// TMEM: S_A 0, O_A 128, S_B 256, O_B 384.  Shared memory: Q_A, Q_B, P, and the
// K and V rings (224 KB).  The GQA group's heads are adjacent in
// the grid, so their K/V tiles are shared through L2.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"
#include "rope.cuh"
#include "tc.cuh"

namespace yoco {

using namespace tc;

constexpr int kFK = 128;                   // keys per tile = query rows per set
constexpr int kFD = 128;                   // head size
constexpr int kFRows = 2 * kFK;            // query rows per CTA
constexpr int kFStages = 2;
constexpr int kFTile = kFK * kFD * 2;      // 32 KB bf16 tile
constexpr int kFHalf = kFTile / 2;         // one 64-column block
constexpr int kFThreads = 320;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleGap2 = 8.f * kLog2e;  // reference moves only when passed by more than e^8

struct FaSmem {
    uint64_t q_full;
    uint64_t kfull[kFStages], kempty[kFStages], vfull[kFStages], vempty[kFStages];  // K and V slots apart
    uint64_t s_full[2], s_free[2];          // per set
    uint64_t p_ready[2][2], pv_done[2][2];  // per set and 64-key half of P
    int walive[2][4];                              // per set and softmax warp, after the tile loop
    uint64_t q_rot[2];                           // per set: Q tile turned (rotary encoding) or as loaded
    float rope_c[2][64], rope_s[2][64], rope_th[2][64];
    uint32_t tmem_base;
    int abort_flag;
    int go[2];
};

constexpr size_t kFTileBytes = (size_t)3 * kFTile + (size_t)kFStages * 2 * kFTile;  // Q_A, Q_B, P + K/V rings
constexpr size_t kFSmem = kFTileBytes + sizeof(FaSmem) + 1024;
static_assert(kFSmem <= 232448, "flash-attention tiles must fit shared memory");

// named barrier (aligned form: the warp is reconverged first, see gret_tc.cu)
__device__ __forceinline__ void fbar(int id, int n) {
    __syncwarp();
    asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(n) : "memory");
}

__device__ __forceinline__ uint32_t fa_tile_chunk(int r, int c) {  // 16-B chunk c (0..15) of row r, SW128
    return (uint32_t)(c >> 3) * kFHalf + (uint32_t)r * 128u + (uint32_t)(((c & 7) ^ (r & 7)) * 16);
}

__device__ __forceinline__ uint32_t fa_pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h2 = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h2);
}

__device__ __forceinline__ float fa_ex2(float x) {  // 2^x, hardware approximation (exact 0 at -inf)
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
    return y;
}

__global__ void __launch_bounds__(kFThreads, 1)
attn_fa_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o, int T, int Hq,
               int Hkv, int64_t p0, float scale, int64_t window, int kv_token_major, int *err, float rope_base,
               const RopeFreq rf) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
    uint8_t *tiles = smem_raw + pad;
    uint8_t *sQ = tiles;                      // Q_A, Q_B (later the output staging tiles)
    uint8_t *sP = tiles + 2 * kFTile;         // P of one set at a time (A(i), B(i), A(i + 1), ...)
    uint8_t *ring = tiles + 3 * kFTile;       // stage s: K at ring + 2 s kFTile, V after it
    FaSmem &sm = *reinterpret_cast<FaSmem *>(tiles + kFTileBytes);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h = blockIdx.x % Hq;
    const int b = blockIdx.x / Hq;
    const int qb = (int)gridDim.y - 1 - (int)blockIdx.y;  // longest rows first
    const int q0 = qb * kFRows;
    const int G = Hq / Hkv;
    const int hk = h / G;            // kv head
    const int64_t pos_lo = p0 + q0;
    const int64_t pos_hi = p0 + min(q0 + kFRows, T) - 1;
    const int64_t key_lo = (window > 0) ? max((int64_t)0, pos_lo - window + 1) : 0;
    const int j_lo = (int)(key_lo / kFK), j_hi = (int)(pos_hi / kFK);
    const int ntiles = j_hi - j_lo + 1;

    if (tid == 0) {
        mbar_init(&sm.q_full, 1);
        for (int s = 0; s < kFStages; ++s) {
            mbar_init(&sm.kfull[s], 1);
            mbar_init(&sm.kempty[s], 1);
            mbar_init(&sm.vfull[s], 1);
            mbar_init(&sm.vempty[s], 1);
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(&sm.s_full[x], 1);
            mbar_init(&sm.s_free[x], 4);   // one arrival per softmax warp of the set: S read out
            for (int hh = 0; hh < 2; ++hh) {
                mbar_init(&sm.p_ready[x][hh], 4);  // one arrival per softmax warp of the set
                mbar_init(&sm.pv_done[x][hh], 1);
            }
            mbar_init(&sm.q_rot[x], 1);
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
            mbar_arrive_expect_tx(&sm.q_full, 2 * kFTile);
            for (int x = 0; x < 2; ++x)
                for (int half = 0; half < 2; ++half)
                    tma_load_4d(sQ + x * kFTile + half * kFHalf, &tm_q, &sm.q_full, half * 64, h, q0 + x * kFK, b);
            // K(i) reuses the slot of K(i - 2) once both S MMAs of tile i - 2 are done, V(i)
            // that of V(i - 2) once both P V MMAs are.  The MMAs free K(i - 1)'s slot before
            // V(i - 2)'s (S_B(i - 1) precedes P_B V(i - 2)), so K runs one tile ahead: K(0),
            // K(1), V(0), K(2), V(1), ...
            int nk = 0, nv = 0;  // tiles whose K / V copy was issued
            auto load = [&](int i, bool is_v) -> bool {
                const int s = i % kFStages;
                const int key0 = (j_lo + i) * kFK;
                uint8_t *st = ring + (size_t)s * 2 * kFTile + (is_v ? kFTile : 0);
                uint64_t *full = is_v ? &sm.vfull[s] : &sm.kfull[s];
                // K/V as {d, key, kv head, b} (a cache) or {d, kv head, key, b} (token-major)
                const int c1 = kv_token_major ? hk : key0, c2 = kv_token_major ? key0 : hk;
                if (i >= kFStages &&
                    !mbar_wait(is_v ? &sm.vempty[s] : &sm.kempty[s], ((i / kFStages) + 1) & 1, abort_flag)) {
                    fail(31);
                    return false;
                }
                mbar_arrive_expect_tx(full, kFTile);
                for (int half = 0; half < 2; ++half)
                    tma_load_4d(st + half * kFHalf, is_v ? &tm_v : &tm_k, full, half * 64, c1, c2, b);
                ++(is_v ? nv : nk);
                return true;
            };
            bool okp = ntiles <= 0 || load(0, false);
            for (int i = 0; i < ntiles && okp; ++i) {
                if (i + 1 < ntiles && !(okp = load(i + 1, false))) break;
                okp = load(i, true);
            }
            // leave no copy in flight (only the last two of each kind can be)
            mbar_wait(&sm.q_full, 0, abort_flag, 200000000ull);
            for (int k = max(0, nk - kFStages); k < nk; ++k)
                mbar_wait(&sm.kfull[k % kFStages], (k / kFStages) & 1, abort_flag, 200000000ull);
            for (int k = max(0, nv - kFStages); k < nv; ++k)
                mbar_wait(&sm.vfull[k % kFStages], (k / kFStages) & 1, abort_flag, 200000000ull);
        }
    } else if (warp == 1) {
        // -------------------------------------------------------------- MMA
        if (lane == 0) {
            const uint32_t id_s = idesc_bf16_f32(kFK, kFK, false, false);  // A = Q (K-major), B = K (K-major)
            const uint32_t id_o = idesc_bf16_f32(kFK, kFD, false, true);   // A = P (K-major), B = V (N-major)
            bool ok = mbar_wait(&sm.q_full, 0, abort_flag);
            // S_X(i) = Q_X K(i)^T into the set's S columns, once the set's softmax warps have
            // read S_X(i - 1) out of them
            auto issue_s = [&](int x, int i) -> bool {
                if (i > 0 && !mbar_wait(&sm.s_free[x], (i - 1) & 1, abort_flag)) return false;
                if (i == 0 && !mbar_wait(&sm.q_rot[x], 0, abort_flag)) return false;  // Q_X as the MMA reads it
                tc_fence_after();
                // descriptors built once and stepped: the address field (bytes / 16, 14 bits)
                // cannot carry out below 256 KB of shared memory
                const uint64_t dq = smem_desc_sw128(smem_u32(sQ + x * kFTile), 16, 1024);
                const uint64_t dk = smem_desc_sw128(smem_u32(ring + (size_t)(i % kFStages) * 2 * kFTile), 16, 1024);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint64_t off = ((kk >> 2) * kFHalf + (kk & 3) * 32) >> 4;
                    mma_ss(tmem + 256 * x, dq + off, dk + off, id_s, kk > 0);
                }
                mma_commit(&sm.s_full[x]);
                return true;
            };
            auto issue_pv = [&](int x, int i) -> bool {  // O_X += P_X(i) V(i), P from shared memory
                // set A's P V is the first use of V(i)
                if (x == 0 && !mbar_wait(&sm.vfull[i % kFStages], (i / kFStages) & 1, abort_flag)) return false;
                const uint64_t dp = smem_desc_sw128(smem_u32(sP), 16, 1024);
                const uint64_t dv = smem_desc_sw128(smem_u32(ring + (size_t)(i % kFStages) * 2 * kFTile + kFTile), kFHalf, 1024);
                // by 64-key halves of P: each half's MMAs go as soon as the set has written it,
                // and its barrier tells the other set when that half of the buffer is free
                for (int hh = 0; hh < 2; ++hh) {
                    if (!mbar_wait(&sm.p_ready[x][hh], i & 1, abort_flag)) return false;
                    tc_fence_after();
#pragma unroll
                    for (int k4 = 0; k4 < 4; ++k4) {
                        const int kk = 4 * hh + k4;
                        mma_ss(tmem + 256 * x + 128, dp + (uint64_t)((hh * kFHalf + k4 * 32) >> 4),
                               dv + (uint64_t)((kk * 2048) >> 4), id_o, (i > 0 || kk > 0));
                    }
                    mma_commit(&sm.pv_done[x][hh]);
                }
                return true;
            };
            // S_A(0), S_B(0), then per tile i: S_A(i + 1), P_A V(i), S_B(i + 1), P_B V(i).  Set B
            // writes P(i) once P_A V(i) is done and set A writes P(i + 1) once P_B V(i) is, so the
            // two P V MMAs alternate on one buffer, and each S sits between them.
            if (ok && ntiles > 0) {
                ok = mbar_wait(&sm.kfull[0], 0, abort_flag) && issue_s(0, 0) && issue_s(1, 0);
                if (ok) mma_commit(&sm.kempty[0]);  // K(0) fully used
            }
            for (int i = 0; i < ntiles && ok; ++i) {
                const bool next = i + 1 < ntiles;
                const int s1 = (i + 1) % kFStages;
                if (next && !(ok = mbar_wait(&sm.kfull[s1], ((i + 1) / kFStages) & 1, abort_flag))) break;
                if (next && !(ok = issue_s(0, i + 1))) break;
                if (!(ok = issue_pv(0, i))) break;
                if (next) {
                    if (!(ok = issue_s(1, i + 1))) break;
                    mma_commit(&sm.kempty[s1]);  // K(i + 1) fully used
                }
                if (!(ok = issue_pv(1, i))) break;
                mma_commit(&sm.vempty[i % kFStages]);  // V(i) fully used
            }
            if (!ok) fail(32);
        }
    } else {
        // ------------------------------------------ softmax, rescale, epilogue
        const int x = (warp - 2) / 4;   // set: A (warps 2-5) or B (6-9)
        const int q4 = warp & 3;        // TMEM lane quarter of this warp
        const int r = q4 * 32 + lane;   // row of the set = TMEM lane
        const int bar_id = 1 + x;
        const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
        const uint32_t colS = 256 * x, colO = 256 * x + 128;
        const int64_t set_lo = p0 + q0 + x * kFK;       // position of the set's first row
        const int64_t pos = set_lo + r;
        const float c2 = scale * kLog2e;
        float m_ref = -INFINITY, l = 0.f;                // base-2 units
        bool alive = true;
        if (rope_base > 0.f) {
            // rotary encoding of this set's Q rows in place: row r at position set_lo + r
            // turns pair i by (set_lo + r) theta_i = base angle (fp64, once per pair) + r theta_i
            if (r == 0) {
                const bool ok = mbar_wait(&sm.q_full, 0, abort_flag);
                if (!ok) fail(36);
                sm.go[x] = ok && !*abort_flag;
            }
            if (r < kFD / 2) {
                const double th = rf.theta[r];
                rope_cs_exact(set_lo, th, sm.rope_c[x][r], sm.rope_s[x][r]);
                sm.rope_th[x][r] = (float)th;
            }
            fbar(bar_id, 128);
            alive = sm.go[x];
            if (alive) {
                uint8_t *qt = sQ + x * kFTile;
#pragma unroll 1
                for (int ch = 0; ch < kFD / 8; ++ch) {  // 16-byte chunk = 4 pairs
                    uint4 *p = reinterpret_cast<uint4 *>(qt + fa_tile_chunk(r, ch));
                    uint4 u = *p;
                    uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int i = ch * 4 + q;
                        float x0 = __uint_as_float(w[q] << 16), x1 = __uint_as_float(w[q] & 0xFFFF0000u);
                        float cj, sj, c, s;
                        rope_cs_offset(r, sm.rope_th[x][i], cj, sj);
                        rope_cs_add(sm.rope_c[x][i], sm.rope_s[x][i], cj, sj, c, s);
                        rope_turn(x0, x1, c, s);
                        w[q] = fa_pack_bf16x2(x0, x1);
                    }
                    *p = make_uint4(w[0], w[1], w[2], w[3]);
                }
                fence_proxy_async_smem();
            }
            fbar(bar_id, 128);
        }
        if (r == 0) mbar_arrive(&sm.q_rot[x]);
        // Per tile, each warp waits for S and announces its rows' P on its own (no
        // named barrier across the set: every thread owns its row)
        for (int i = 0; i < ntiles && alive; ++i) {
            bool okw = true;
            if (lane == 0) {
                okw = mbar_wait(&sm.s_full[x], i & 1, abort_flag);
                if (!okw) fail(33);
                okw = okw && !*abort_flag;
            }
            if (__shfl_sync(0xffffffffu, okw ? 1 : 0, 0) == 0) {
                alive = false;
                break;
            }
            tc_fence_after();
            const uint32_t s_t = tmem + colS + lane_base;
            uint32_t sv[128];
#pragma unroll
            for (int cb = 0; cb < 4; ++cb) tmem_ld32(s_t + cb * 32, *reinterpret_cast<uint32_t(*)[32]>(sv + 32 * cb));
            tmem_wait_ld();
            // S is in registers: the MMA may write S(i + 1) over it
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.s_free[x]);
            const int64_t key0 = (int64_t)(j_lo + i) * kFK;
            // every row of the set sees every key of this tile: no per-element mask
            const bool full = (key0 + kFK - 1 <= set_lo) && (window <= 0 || key0 >= set_lo + kFK - 1 - window + 1);
            // maximum of the raw scores (the scale is positive: it is applied once, to the
            // maximum, and folded into each exponent's argument below), in four chains
            float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
            if (full) {
#pragma unroll
                for (int c = 0; c < kFK; c += 2)
                    mq[(c >> 1) & 3] = fmax3(mq[(c >> 1) & 3], __uint_as_float(sv[c]), __uint_as_float(sv[c + 1]));
            } else {
                // the keys this row sees form one run [lo_c, hi_c) of the tile, held as 4 x 32 bits
                const int64_t first = (window > 0) ? pos - window + 1 : 0;
                const int lo_c = (int)max((int64_t)0, min((int64_t)kFK, first - key0));
                const int hi_c = (int)max((int64_t)0, min((int64_t)kFK, pos + 1 - key0));
                uint32_t bits[4];
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    const int lo = min(max(lo_c - 32 * w, 0), 32), hi = min(max(hi_c - 32 * w, 0), 32);
                    const uint32_t below_hi = (hi >= 32) ? 0xffffffffu : ((1u << hi) - 1u);
                    const uint32_t below_lo = (lo >= 32) ? 0xffffffffu : ((1u << lo) - 1u);
                    bits[w] = below_hi & ~below_lo;
                }
#pragma unroll
                for (int c = 0; c < kFK; c += 2) {
                    const float v0 = (bits[c >> 5] & (1u << (c & 31))) ? __uint_as_float(sv[c]) : -INFINITY;
                    const float v1 = (bits[c >> 5] & (2u << (c & 31))) ? __uint_as_float(sv[c + 1]) : -INFINITY;
                    sv[c] = __float_as_uint(v0);
                    sv[c + 1] = __float_as_uint(v1);
                    mq[(c >> 1) & 3] = fmax3(mq[(c >> 1) & 3], v0, v1);
                }
            }
            const float mt = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3])) * c2;  // -inf stays -inf
            // move the reference maximum only when this tile passes it by more than the gap
            float alpha = 1.f;
            const bool move = (mt > m_ref + kRescaleGap2) || (m_ref == -INFINITY && mt > -INFINITY);
            if (move) {
                alpha = (m_ref == -INFINITY) ? 0.f : fa_ex2(m_ref - mt);
                m_ref = mt;
            }
            const float mu = (m_ref == -INFINITY) ? 0.f : m_ref;  // a row with nothing seen yet: every p is 0
            // P as packed bf16 in registers (keys 2c, 2c+1 in word c): per key pair both exponent
            // arguments s c2 - mu in one packed FMA, the row sum in a packed accumulator
            // (masked scores are -inf and give exactly 0)
            const uint64_t c2x2 = f2_pack(c2, c2), nmu2 = f2_pack(-mu, -mu);
            uint64_t acc2 = f2_pack(0.f, 0.f);
            uint32_t pk[kFK / 2];
#pragma unroll
            for (int c = 0; c < kFK / 2; ++c) {
                float x0, x1;
                f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[2 * c]), __uint_as_float(sv[2 * c + 1])), c2x2, nmu2),
                          x0, x1);
                const float e0 = fa_ex2(x0), e1 = fa_ex2(x1);
                acc2 = f2_add(acc2, f2_pack(e0, e1));
                pk[c] = fa_pack_bf16x2(e0, e1);
            }
            float ls0, ls1;
            f2_unpack(acc2, ls0, ls1);
            const float ls = ls0 + ls1;
            l = fmaf(l, alpha, ls);
            // O_X holds tiles < i; rows whose reference moved rescale it before P V of tile i
            // (the whole warp takes part: TMEM loads and stores are warp-wide)
            if (i > 0 && __any_sync(0xffffffffu, move)) {
                bool ok = true;
                if (lane == 0) ok = mbar_wait(&sm.pv_done[x][1], (i - 1) & 1, abort_flag);  // all of P V(i - 1)
                ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                if (!ok) {
                    if (lane == 0) fail(34);
                } else {
                    tc_fence_after();
                    const uint32_t o_t = tmem + colO + lane_base;
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
            // each 64-key half of the P buffer is free once the other set's P V has read that
            // half: set A's P(i) follows P_B V(i - 1), set B's P(i) follows P_A V(i)
            bool okb = true;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                if (x == 1 || i > 0) {
                    bool ok = true;
                    if (lane == 0) ok = mbar_wait(&sm.pv_done[1 - x][hh], (x == 0 ? i - 1 : i) & 1, abort_flag);
                    if (__shfl_sync(0xffffffffu, ok ? 1 : 0, 0) == 0) {
                        okb = false;
                        break;
                    }
                }
#pragma unroll
                for (int c8 = 0; c8 < kFK / 16; ++c8) {  // 16-byte chunk ch = keys 8 ch .. 8 ch + 7
                    const int ch = hh * (kFK / 16) + c8;
                    *reinterpret_cast<uint4 *>(sP + fa_tile_chunk(r, ch)) =
                        make_uint4(pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
                }
                fence_proxy_async_smem();  // P as the tensor cores read it
                tc_fence_before();
                __syncwarp();  // this warp's rows of this half of P (and rescaled O) are written
                if (lane == 0) mbar_arrive(&sm.p_ready[x][hh]);
            }
            if (!okb) {
                if (lane == 0) fail(37);
                alive = false;
                break;
            }
        }
        // the set agrees on going on: a warp that gave up stops the epilogue for all four
        if (lane == 0) sm.walive[x][q4] = alive ? 1 : 0;
        fbar(bar_id, 128);
        alive = sm.walive[x][0] && sm.walive[x][1] && sm.walive[x][2] && sm.walive[x][3];
        // epilogue: o = O / l as bf16, staged in this set's Q tile (free: every S MMA is done)
        if (alive && ntiles > 0) {
            if (r == 0) {
                const bool ok = mbar_wait(&sm.pv_done[x][1], (ntiles - 1) & 1, abort_flag);
                if (!ok) fail(35);
                sm.go[x] = ok && !*abort_flag;
            }
            fbar(bar_id, 128);
            if (sm.go[x]) {
                tc_fence_after();
                uint8_t *stg = sQ + x * kFTile;
                const float inv = (l > 0.f) ? 1.f / l : 0.f;
                const uint32_t o_t = tmem + colO + lane_base;
#pragma unroll 1
                for (int cb = 0; cb < 4; ++cb) {
                    uint32_t ov[32];
                    tmem_ld32(o_t + cb * 32, ov);
                    tmem_wait_ld();
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        *reinterpret_cast<uint4 *>(stg + fa_tile_chunk(r, cb * 4 + q)) = make_uint4(
                            fa_pack_bf16x2(__uint_as_float(ov[8 * q]) * inv, __uint_as_float(ov[8 * q + 1]) * inv),
                            fa_pack_bf16x2(__uint_as_float(ov[8 * q + 2]) * inv, __uint_as_float(ov[8 * q + 3]) * inv),
                            fa_pack_bf16x2(__uint_as_float(ov[8 * q + 4]) * inv, __uint_as_float(ov[8 * q + 5]) * inv),
                            fa_pack_bf16x2(__uint_as_float(ov[8 * q + 6]) * inv, __uint_as_float(ov[8 * q + 7]) * inv));
                }
                tc_fence_before();
                fence_proxy_async_smem();
                fbar(bar_id, 128);
                if (r == 0 && q0 + x * kFK < T) {  // rows past T are not written
                    tma_store_4d(&tm_o, stg, 0, h, q0 + x * kFK, b);
                    tma_store_4d(&tm_o, stg + kFHalf, 64, h, q0 + x * kFK, b);
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

static cudaError_t fa_run(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv, const CUtensorMap &mo,
                          int B, int T, int Hq, int Hkv, int64_t p0, float scale, int64_t window, int kv_token_major,
                          int *err, float rope_base, cudaStream_t st) {
    cudaError_t e = cudaFuncSetAttribute(attn_fa_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kFSmem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(B * Hq), (unsigned)((T + kFRows - 1) / kFRows));
    cfg.blockDim = dim3(kFThreads);
    cfg.dynamicSmemBytes = kFSmem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    count_launches(1);
    return cudaLaunchKernelEx(&cfg, attn_fa_kernel, mq, mk, mv, mo, T, Hq, Hkv, p0, scale, window, kv_token_major, err,
                              rope_base, make_rope_freq(rope_base, kFD));
}

// [B, rows, H, 128] token-major bf16 as {d, H, rows, B}, box {64, 1, 128, 1}
static bool fa_token_major_map(CUtensorMap *m, const void *ptr, int B, int64_t rows, int H) {
    const cuuint64_t dims[4] = {(cuuint64_t)kFD, (cuuint64_t)H, (cuuint64_t)rows, (cuuint64_t)B};
    const cuuint64_t strides[3] = {(cuuint64_t)kFD * 2, (cuuint64_t)H * kFD * 2, (cuuint64_t)rows * H * kFD * 2};
    const cuuint32_t box[4] = {64, 1, (cuuint32_t)kFK, 1};
    return fa_map(m, 4, ptr, dims, strides, box);
}

cudaError_t attn_fa_launch(const AttnArgs &a, int64_t window, int *err, cudaStream_t st) {
    const int64_t keys = a.p0 + a.T;
    CUtensorMap mq, mk, mv, mo;
    // K, V: cache [B, Hkv, cap, d] viewed with `keys` rows as {d, key, kv head, b}, box {64, 128, 1, 1}
    const cuuint64_t kd[4] = {(cuuint64_t)kFD, (cuuint64_t)keys, (cuuint64_t)a.Hkv, (cuuint64_t)a.B};
    const cuuint64_t ks[3] = {(cuuint64_t)kFD * 2, (cuuint64_t)a.cap * kFD * 2, (cuuint64_t)a.Hkv * a.cap * kFD * 2};
    const cuuint32_t kbox[4] = {64, (cuuint32_t)kFK, 1, 1};
    if (!fa_token_major_map(&mq, a.Q, a.B, a.T, a.Hq) || !fa_token_major_map(&mo, a.O, a.B, a.T, a.Hq) ||
        !fa_map(&mk, 4, a.kc, kd, ks, kbox) || !fa_map(&mv, 4, a.vc, kd, ks, kbox))
        return cudaErrorInvalidValue;
    return fa_run(mq, mk, mv, mo, a.B, a.T, a.Hq, a.Hkv, a.p0, a.scale, window, 0, err, a.rope_base, st);
}

cudaError_t swa_fa_launch(const void *q, const void *k, const void *v, void *o, int B, int N, int Hq, int Hkv,
                          int64_t window, float scale, int *err, cudaStream_t st) {
    CUtensorMap mq, mk, mv, mo;
    if (!fa_token_major_map(&mq, q, B, N, Hq) || !fa_token_major_map(&mo, o, B, N, Hq) ||
        !fa_token_major_map(&mk, k, B, N, Hkv) || !fa_token_major_map(&mv, v, B, N, Hkv))
        return cudaErrorInvalidValue;
    return fa_run(mq, mk, mv, mo, B, N, Hq, Hkv, 0, scale, window, 1, err, 0.0f, st);
}

}  // namespace yoco_host

YOCO_DEBUG_TU(attn_fa)
