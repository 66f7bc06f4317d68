// swa.cu -- the ring cache of the sliding-window self-decoder (paper Section 3.2:
// with a window of C keys the cache holds only the last C tokens, so its size is
// constant however long the sequence grows).  Token at position p lives in slot
// p % C of a [B, Hkv, C, d] ring; the decode attention reads the filled slots in
// any order (softmax does not depend on the order of its keys).
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace yoco {

// one thread per 16 bytes of one (token, b, kv head) row of k or v
__global__ void swa_ring_write_kernel(const uint8_t *__restrict__ k, const uint8_t *__restrict__ v,
                                      uint8_t *__restrict__ rk, uint8_t *__restrict__ rv, int B, int N, int Hkv,
                                      int row_bytes, int window, int64_t tok0, int n, int64_t pos0) {
    const int vec = row_bytes / 16;
    const int64_t total = (int64_t)2 * n * B * Hkv * vec;
    for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < total; e += (int64_t)gridDim.x * blockDim.x) {
        int64_t r = e;
        const int c = (int)(r % vec);
        r /= vec;
        const int hk = (int)(r % Hkv);
        r /= Hkv;
        const int b = (int)(r % B);
        r /= B;
        const int i = (int)(r % n);
        const int which = (int)(r / n);  // 0: k, 1: v
        const int64_t tok = tok0 + i;
        const int64_t slot = (pos0 + i) % window;
        if (!YOCO_DCHECK(tok < N && slot >= 0 && slot < window, 0x5E)) continue;
        const uint8_t *src = (which ? v : k) + (((size_t)b * N + tok) * Hkv + hk) * (size_t)row_bytes;
        uint8_t *dst = (which ? rv : rk) + (((size_t)b * Hkv + hk) * window + slot) * (size_t)row_bytes;
        reinterpret_cast<uint4 *>(dst)[c] = reinterpret_cast<const uint4 *>(src)[c];
    }
}

}  // namespace yoco

namespace yoco_host {
using namespace yoco;

cudaError_t swa_ring_write(const void *k, const void *v, void *rk, void *rv, int B, int N, int Hkv, int d,
                           int window, int64_t tok0, int n, int64_t pos0, yoco_dtype dt, cudaStream_t st) {
    if (n <= 0) return cudaSuccess;
    const int row_bytes = d * (dt == YOCO_BF16 ? 2 : 4);
    const int64_t total = (int64_t)2 * n * B * Hkv * (row_bytes / 16);
    const int blocks = (int)std::min<int64_t>((total + 255) / 256, (int64_t)device_sm_count() * 8);
    count_launches(1);
    swa_ring_write_kernel<<<blocks, 256, 0, st>>>((const uint8_t *)k, (const uint8_t *)v, (uint8_t *)rk,
                                                  (uint8_t *)rv, B, N, Hkv, row_bytes, window, tok0, n, pos0);
    return cudaGetLastError();
}

}  // namespace yoco_host

YOCO_DEBUG_TU(swa)
