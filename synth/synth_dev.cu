// synth_dev.cu -- device copy of the seeded input generator in synth/__init__.py.
// Counter based: element i of stream `stream` under `seed` depends on nothing else,
// so a full-size tensor made here and a slice regenerated on the host agree.  It
// holds none of the method's arithmetic and is not part of libyoco.
#include <cuda_runtime.h>
#include <stdint.h>

#define SYNTH_API extern "C" __attribute__((visibility("default")))

__host__ __device__ static inline uint64_t splitmix64(uint64_t x) {
    x += 0x9E3779B97F4A7C15ull;
    x = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9ull;
    x = (x ^ (x >> 27)) * 0x94D049BB133111EBull;
    return x ^ (x >> 31);
}

static uint64_t stream_key(uint64_t seed, uint64_t stream) { return splitmix64(splitmix64(seed) ^ stream); }

__device__ static inline double normal_at(uint64_t key, uint64_t i, double mean, double stdv) {
    uint64_t a = splitmix64(key + 2ull * i);
    uint64_t b = splitmix64(key + 2ull * i + 1ull);
    double u1 = (double)((a >> 11) + 1ull) * 0x1.0p-53;
    double u2 = (double)(b >> 11) * 0x1.0p-53;
    double z = sqrt(-2.0 * log(u1)) * cos(6.283185307179586 * u2);
    return mean + stdv * z;
}

// fp64 -> bf16 bits, nearest-even: fp32 round-to-odd, then nearest-even on the bits
__device__ static inline uint16_t to_bf16_bits(double x) {
    float t = __double2float_rz(x);
    uint32_t bits = __float_as_uint(t);
    if ((double)t != x) bits |= 1u;
    bits += 0x7FFFu + ((bits >> 16) & 1u);
    return (uint16_t)(bits >> 16);
}

__global__ void normal_bf16_kernel(uint16_t *out, int64_t n, uint64_t key, double mean, double stdv, int64_t start) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
        out[i] = to_bf16_bits(normal_at(key, (uint64_t)(start + i), mean, stdv));
}

__global__ void normal_f32_kernel(float *out, int64_t n, uint64_t key, double mean, double stdv, int64_t start) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
        out[i] = (float)normal_at(key, (uint64_t)(start + i), mean, stdv);
}

static int grid_for(int64_t n) {
    int64_t g = (n + 255) / 256;
    return (int)(g > 152 * 32 ? 152 * 32 : (g < 1 ? 1 : g));
}

SYNTH_API int synth_normal_bf16(void *out, int64_t n, uint64_t seed, uint64_t stream, double mean, double stdv,
                                int64_t start, void *cuda_stream) {
    if (n <= 0) return 0;
    normal_bf16_kernel<<<grid_for(n), 256, 0, (cudaStream_t)cuda_stream>>>((uint16_t *)out, n, stream_key(seed, stream),
                                                                            mean, stdv, start);
    return (int)cudaGetLastError();
}

SYNTH_API int synth_normal_f32(void *out, int64_t n, uint64_t seed, uint64_t stream, double mean, double stdv,
                               int64_t start, void *cuda_stream) {
    if (n <= 0) return 0;
    normal_f32_kernel<<<grid_for(n), 256, 0, (cudaStream_t)cuda_stream>>>((float *)out, n, stream_key(seed, stream),
                                                                           mean, stdv, start);
    return (int)cudaGetLastError();
}
