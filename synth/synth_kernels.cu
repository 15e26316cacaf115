// synth_kernels.cu -- the seeded input generator of synth/__init__.py, on the GPU and as fast
// host code.  Same definition, same bits: counter-based SplitMix64 (Steele, Lea & Flood,
// OOPSLA 2014), Irwin-Hall(12) normal approximation, uniform from the top 24 bits; double
// arithmetic rounded operation by operation (no fused multiply-add), then float32, then
// (for bfloat16) round-to-nearest-even.  Holds nothing of the convolution's arithmetic.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

namespace {

constexpr uint64_t kGolden = 0x9E3779B97F4A7C15ull;

__host__ __device__ inline uint64_t mix64(uint64_t z)
{
    z ^= z >> 30;
    z *= 0xBF58476D1CE4E5B9ull;
    z ^= z >> 27;
    z *= 0x94D049BB133111EBull;
    z ^= z >> 31;
    return z;
}

__host__ __device__ inline uint64_t tensor_key(uint64_t seed, unsigned tensor_id)
{
    return mix64(seed + (uint64_t)(tensor_id + 1) * kGolden);
}

#if defined(__CUDA_ARCH__)
#define DMUL(a, b) __dmul_rn((a), (b))
#define DADD(a, b) __dadd_rn((a), (b))
#else
#define DMUL(a, b) ((a) * (b))
#define DADD(a, b) ((a) + (b))
#endif

// dist 0: normal, sigma = p1 (p0 must be 0).  dist 1: uniform [p0, p1).
__host__ __device__ inline double value_f64(uint64_t key, int dist, double p0, double p1, uint64_t e)
{
    if (dist == 0) {
        int64_t S = 0;
        for (int j = 0; j < 3; ++j) {
            const uint64_t z = mix64(key + (e * 3 + (uint64_t)j + 1) * kGolden);
            for (int q = 0; q < 4; ++q) S += (int64_t)((z >> (16 * q)) & 0xFFFFull);
        }
        const double v = (double)(S - 393210) / 65536.0;
        return DMUL(v, p1);
    }
    const uint64_t z = mix64(key + (e + 1) * kGolden);
    const double u = (double)(z >> 40) / 16777216.0;
    const double span = p1 - p0;
    return DADD(p0, DMUL(span, u));
}

inline uint16_t f32_to_bf16_bits_host(float f)
{
    uint32_t b;
    memcpy(&b, &f, 4);
    const uint32_t rnd = ((b >> 16) & 1u) + 0x7FFFu;
    return (uint16_t)((b + rnd) >> 16);
}

__global__ void fill_kernel(void* out, int dtype, int dist, uint64_t key, long long offset, long long count, double p0,
                            double p1)
{
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < count;
         i += (long long)gridDim.x * blockDim.x) {
        const double v = value_f64(key, dist, p0, p1, (uint64_t)(offset + i));
        const float f = __double2float_rn(v);
        if (dtype == 0)
            static_cast<float*>(out)[i] = f;
        else
            static_cast<__nv_bfloat16*>(out)[i] = __float2bfloat16_rn(f);
    }
}

}  // namespace

extern "C" {

// Fill `count` consecutive elements (global indices offset .. offset+count-1) on the GPU.
// dtype 0 = float32, 1 = bfloat16.  Returns a cudaError_t code.
int synth_fill_device(void* out, int dtype, int dist, unsigned long long seed, unsigned tensor_id, long long offset,
                      long long count, double p0, double p1, void* stream)
{
    if (count <= 0) return 0;
    long long blocks = (count + 255) / 256;
    if (blocks > 152 * 32) blocks = 152 * 32;
    fill_kernel<<<(unsigned)blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(out, dtype, dist,
                                                                                  tensor_key(seed, tensor_id), offset,
                                                                                  count, p0, p1);
    return (int)cudaGetLastError();
}

// Host version at arbitrary global indices: out[i] = value(idx[i]) as float32 or bf16 bits.
void synth_values_host(void* out, int dtype, int dist, unsigned long long seed, unsigned tensor_id,
                       const long long* idx, long long n, double p0, double p1)
{
    const uint64_t key = tensor_key(seed, tensor_id);
    for (long long i = 0; i < n; ++i) {
        const float f = (float)value_f64(key, dist, p0, p1, (uint64_t)idx[i]);
        if (dtype == 0)
            static_cast<float*>(out)[i] = f;
        else
            static_cast<uint16_t*>(out)[i] = f32_to_bf16_bits_host(f);
    }
}

}  // extern "C"
