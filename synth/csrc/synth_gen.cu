// Device twin of synth/cpu.py: the same counter-based values (splitmix64 words, twelve-term
// Irwin-Hall sum, round-to-nearest-even bf16), the same planted keys, written straight into
// device memory so that multi-GB workloads never cross the host link.  Input generation only:
// nothing of the token-dropping method is computed here.
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ull;

__device__ __forceinline__ uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

__device__ __forceinline__ uint64_t word(uint64_t key, uint64_t idx, int k) {
    return mix64(key + (idx * 3ull + static_cast<uint64_t>(k + 1)) * kGamma);
}

__device__ __forceinline__ uint16_t f32_to_bf16_rne(float x) {
    const uint32_t b = __float_as_uint(x);
    return static_cast<uint16_t>((b + 0x7FFFu + ((b >> 16) & 1u)) >> 16);
}

__device__ __forceinline__ float bf16_to_f32(uint16_t h) { return __uint_as_float(static_cast<uint32_t>(h) << 16); }

__device__ __forceinline__ uint16_t normal_bf16(uint64_t key, uint64_t idx) {
    const uint64_t lanes = 0x0000FFFF0000FFFFull;
    uint64_t acc = 0;
#pragma unroll
    for (int k = 0; k < 3; ++k) {
        const uint64_t w = word(key, idx, k);
        acc += (w & lanes) + ((w >> 16) & lanes);
    }
    const uint64_t s = (acc & 0xFFFFFFFFull) + (acc >> 32);
    const float z = static_cast<float>(static_cast<int64_t>(s) - 393210) * (1.0f / 65536.0f);
    return f32_to_bf16_rne(z);
}

__global__ void normal_kernel(uint16_t* out, uint64_t key, uint64_t start, uint64_t count) {
    for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < count; i += (uint64_t)gridDim.x * blockDim.x)
        out[i] = normal_bf16(key, start + i);
}

__global__ void slots_kernel(int64_t* out, uint64_t key, uint64_t start, uint64_t count) {
    for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < count; i += (uint64_t)gridDim.x * blockDim.x)
        out[i] = static_cast<int64_t>(word(key, start + i, 0) & ((1ull << 40) - 1));
}

__device__ __forceinline__ int request_of(const int32_t* cu, int R, int64_t t) {
    int lo = 0, hi = R;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (cu[mid] <= t) lo = mid; else hi = mid;
    }
    return lo;
}

__global__ void positions_kernel(int64_t* out, const int32_t* cu, int R, int64_t T) {
    for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < T; t += (int64_t)gridDim.x * blockDim.x)
        out[t] = t - cu[request_of(cu, R, t)];
}

// K rows of sink tokens (local index < sink_tokens) are scaled by sink_scale; K rows of hot tokens
// get + shift * u[r, kh, :] in fp32, then round to bf16 (same two roundings as the numpy twin).
__global__ void plant_kernel(uint16_t* K, const int32_t* cu, int R, int64_t T, int Hkv, int dk,
                             const uint8_t* hot_tok, const float* u, int sink_tokens, float sink_scale, float shift) {
    const int64_t row_elems = (int64_t)Hkv * dk;
    for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < T * row_elems;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int64_t t = e / row_elems;
        const int r = request_of(cu, R, t);
        const int64_t loc = t - cu[r];
        const bool sink = loc < sink_tokens;
        const bool hot = hot_tok[t] != 0;
        if (!sink && !hot) continue;
        float v = bf16_to_f32(K[e]);
        if (sink) v = bf16_to_f32(f32_to_bf16_rne(__fmul_rn(v, sink_scale)));
        if (hot) {
            const int64_t he = e - t * row_elems;               // kh * dk + d
            v = bf16_to_f32(f32_to_bf16_rne(__fadd_rn(v, __fmul_rn(shift, u[(int64_t)r * row_elems + he]))));
        }
        K[e] = f32_to_bf16_rne(v);
    }
}

int grid_for(uint64_t n) {
    uint64_t g = (n + 255) / 256;
    return static_cast<int>(g > 65535ull * 16 ? 65535ull * 16 : (g == 0 ? 1 : g));
}

}  // namespace

extern "C" int synth_normal_bf16(void* out, uint64_t key, uint64_t start, uint64_t count, void* stream) {
    if (count == 0) return 0;
    normal_kernel<<<grid_for(count), 256, 0, static_cast<cudaStream_t>(stream)>>>(static_cast<uint16_t*>(out), key,
                                                                                  start, count);
    return static_cast<int>(cudaGetLastError());
}

extern "C" int synth_slots(void* out, uint64_t key, uint64_t start, uint64_t count, void* stream) {
    if (count == 0) return 0;
    slots_kernel<<<grid_for(count), 256, 0, static_cast<cudaStream_t>(stream)>>>(static_cast<int64_t*>(out), key,
                                                                                 start, count);
    return static_cast<int>(cudaGetLastError());
}

extern "C" int synth_positions(void* out, const void* cu, int R, int64_t T, void* stream) {
    if (T == 0) return 0;
    positions_kernel<<<grid_for(T), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<int64_t*>(out), static_cast<const int32_t*>(cu), R, T);
    return static_cast<int>(cudaGetLastError());
}

extern "C" int synth_plant_k(void* K, const void* cu, int R, int64_t T, int Hkv, int dk, const void* hot_tok,
                             const void* u, int sink_tokens, float sink_scale, float shift, void* stream) {
    if (T == 0) return 0;
    plant_kernel<<<grid_for((uint64_t)T * Hkv * dk), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<uint16_t*>(K), static_cast<const int32_t*>(cu), R, T, Hkv, dk,
        static_cast<const uint8_t*>(hot_tok), static_cast<const float*>(u), sink_tokens, sink_scale, shift);
    return static_cast<int>(cudaGetLastError());
}
