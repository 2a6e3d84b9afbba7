// GPU twin of the seeded input generator in synth.py (same definitions, bit
// for bit): stream `key` at counter i is mix(key + (i + 1) * GAMMA), with mix
// the SplitMix64 output function (Steele, Lea & Flood, OOPSLA 2014). Holds
// input distributions only; none of the CSA2 method's arithmetic lives here.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ull;
constexpr int kMaxStreams = 64;
enum Kind { NORMAL_F32 = 0, NORMAL_BF16 = 1, E2M1_BYTES = 2, SCALE_POW2_BYTES = 3, W_POW2_F32 = 4 };

struct Keys {
    uint64_t k[kMaxStreams];
};

__device__ __forceinline__ uint64_t mix(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

__device__ __forceinline__ uint64_t draw(uint64_t key, uint64_t c) { return mix(key + (c + 1) * kGamma); }

__device__ __forceinline__ float normal(uint64_t key, uint64_t c) {
    const uint64_t a = draw(key, 2 * c), b = draw(key, 2 * c + 1);
    int s = 0;
#pragma unroll
    for (int sh = 0; sh < 64; sh += 16) s += (int)((a >> sh) & 0xFFFF) + (int)((b >> sh) & 0xFFFF);
    // 1/sqrt(32*(65536^2-1)/12) in fp32 (bits 0x371CC471): unit variance
    return __fmul_rn(__int2float_rn(2 * s - 8 * 65535), __uint_as_float(0x371CC471u));
}

__constant__ uint8_t kE2M1Codes15[15] = {0xF, 0xE, 0xD, 0xC, 0xB, 0xA, 0x9, 0x0,
                                         0x1, 0x2, 0x3, 0x4, 0x5, 0x6, 0x7};

__global__ void k_fill(int kind, Keys keys, int n_streams, uint64_t counter0, int64_t n_per,
                       void* out, int64_t stride) {
    const int64_t total = (int64_t)n_streams * n_per;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int s = (int)(e / n_per);
        const int64_t i = e - (int64_t)s * n_per;
        const uint64_t key = keys.k[s], c = counter0 + (uint64_t)i;
        const int64_t o = (int64_t)s * stride + i;
        switch (kind) {
            case NORMAL_F32: static_cast<float*>(out)[o] = normal(key, c); break;
            case NORMAL_BF16:
                static_cast<__nv_bfloat16*>(out)[o] = __float2bfloat16_rn(normal(key, c));
                break;
            case E2M1_BYTES: {
                const uint64_t x = draw(key, c);
                const uint32_t lo = (uint32_t)(((x & 0xFFFF) * 15) >> 16);
                const uint32_t hi = (uint32_t)((((x >> 16) & 0xFFFF) * 15) >> 16);
                static_cast<uint8_t*>(out)[o] = (uint8_t)(kE2M1Codes15[lo] | (kE2M1Codes15[hi] << 4));
                break;
            }
            case SCALE_POW2_BYTES:
                static_cast<uint8_t*>(out)[o] = (draw(key, c) & 1) ? 0x40 : 0x38;
                break;
            case W_POW2_F32: {
                const int u = (int)(draw(key, c) & 3) - 2;
                static_cast<float*>(out)[o] = ldexpf(1.0f, u);
                break;
            }
        }
    }
}

}  // namespace

// Fills out[s * stride + i] (elements of the kind's type) for s < n_streams,
// i < n_per_stream, with the value of stream keys[s] at counter counter0 + i.
// keys is a HOST array. Returns 0, or 1 on bad arguments, 2 on a launch error.
extern "C" int csa2synth_fill(int kind, const uint64_t* keys, int n_streams, uint64_t counter0,
                              int64_t n_per_stream, void* out, int64_t stride, void* stream) {
    if (n_streams < 0 || n_streams > kMaxStreams || n_per_stream < 0 || kind < 0 || kind > 4)
        return 1;
    if (n_streams == 0 || n_per_stream == 0) return 0;
    if (!keys || !out) return 1;
    Keys k;
    for (int s = 0; s < n_streams; ++s) k.k[s] = keys[s];
    const int64_t total = (int64_t)n_streams * n_per_stream;
    int64_t blocks = (total + 255) / 256;
    if (blocks > 152 * 64) blocks = 152 * 64;
    k_fill<<<(unsigned)blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(
        kind, k, n_streams, counter0, n_per_stream, out, stride);
    return cudaGetLastError() == cudaSuccess ? 0 : 2;
}
