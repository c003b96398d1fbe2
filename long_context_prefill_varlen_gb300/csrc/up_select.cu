// up_select_topp and up_make_cu_blocks: top-p block selection of UniPrefill ("UniPrefill:
// Universal Long-Context Prefill Acceleration via Block-wise Dynamic Sparsification",
// arXiv 2605.06221, section 3.3 Eq. 5 with the forced sink/window tokens, and the top-p kernel of
// section 3.5 with the packed sort key of Eq. 14).
//
// One CTA per request, everything in shared memory, no CPU round trip:
//   1. key_g = (phi(b_g) << 32) | g for the request's blocks (phi(x) = bits(x) ^ 0x80000000 for
//      x >= 0; scores are non-negative sums of probabilities, so the sign bit decides phi).
//   2. LSD radix sort of the 64-bit keys, descending, 4-bit digits, stable: the low word holds g
//      (< 2^16), so only its low 16 bits and the 32 high bits carry information; digit passes
//      above the block-index range are identity permutations and are skipped.
//   3. inclusive prefix sum of the sorted scores in fp64 (fixed tree), k* = 1 + #{k : cum_k < p*total}.
//   4. ranked flags by block index, then the byte masks: block(i) ranked, or i < A, or i >= N - n.
#include <stdint.h>

#include "up_internal.cuh"

namespace up {
namespace select {

constexpr int kThreads = 512;
constexpr int kMaxIpt = UP_MAX_BLOCKS_PER_REQUEST / kThreads;   // 16 keys per thread
constexpr int kDigits = 16;

__device__ __forceinline__ uint64_t pack_key(float b, uint32_t g) {
    const uint32_t bits = __float_as_uint(b);
    const uint32_t phi = (bits & 0x80000000u) ? ~bits : (bits ^ 0x80000000u);
    return (static_cast<uint64_t>(phi) << 32) | g;
}

// exclusive scan of one value per thread over the 512 threads, fixed association (fp64 or int)
template <typename T>
__device__ __forceinline__ T block_exclusive_scan(T v, T* sh, T* total) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    T x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        T y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    T excl = __shfl_up_sync(0xffffffffu, x, 1);
    if (lane == 0) excl = T(0);
    if (lane == 31) sh[w] = x;
    __syncthreads();
    if (w == 0) {
        T s = lane < kThreads / 32 ? sh[lane] : T(0);
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            T y = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o) s += y;
        }
        T e = __shfl_up_sync(0xffffffffu, s, 1);
        if (lane == 0) e = T(0);
        if (lane < kThreads / 32) sh[32 + lane] = e;          // exclusive warp offsets
        if (lane == kThreads / 32 - 1) sh[64] = s;             // grand total
    }
    __syncthreads();
    const T before = sh[32 + w] + excl;
    *total = sh[64];
    __syncthreads();
    return before;
}

__global__ void __launch_bounds__(kThreads) select_kernel(const float* __restrict__ bs, const int32_t* __restrict__ cb,
                                                          const int32_t* __restrict__ cu, int R, int T, int64_t nb_cap,
                                                          int G, int n, int A, double p, uint8_t* block_keep,
                                                          uint8_t* token_keep, int32_t* kstar, int32_t* status) {
    extern __shared__ __align__(16) uint8_t sm[];
    uint64_t* keys = reinterpret_cast<uint64_t*>(sm);                              // [8192]
    uint64_t* alt = keys + UP_MAX_BLOCKS_PER_REQUEST;                              // [8192]
    uint32_t* cnt = reinterpret_cast<uint32_t*>(alt + UP_MAX_BLOCKS_PER_REQUEST);  // [16][512]
    uint8_t* ranked = reinterpret_cast<uint8_t*>(cnt + kDigits * kThreads);        // [8192]
    __shared__ double shd[65];
    __shared__ int shi[65];
    __shared__ double s_total;
    __shared__ int s_bad;

    const int r = blockIdx.x, tid = threadIdx.x;
    const int c0 = cu[r], c1 = cu[r + 1];
    const int N = c1 - c0;
    const int nb = N > 0 ? (N + G - 1) / G : 0;
    if (tid == 0) {
        int bad = 0;
        if ((r == 0 && c0 != 0) || c1 < c0 || c1 > T || (r == R - 1 && c1 != T)) bad = UP_DEV_BAD_CU_SEQLENS;
        else if ((r == 0 && cb[0] != 0) || cb[r + 1] - cb[r] != nb || (int64_t)cb[r + 1] > nb_cap) bad = UP_DEV_BAD_CU_BLOCKS;
        else if (nb > UP_MAX_BLOCKS_PER_REQUEST) bad = UP_DEV_TOO_MANY_BLOCKS;
        s_bad = bad;
        if (bad) set_status(status, bad);
    }
    __syncthreads();
    if (s_bad) return;
    if (nb == 0) {
        if (tid == 0) kstar[r] = 0;
        return;
    }
    const int b0 = cb[r];
    const int ipt = (nb + kThreads - 1) / kThreads;      // keys per thread, contiguous
    const int k0 = tid * ipt;

    // 1. packed keys (padding slots get key 0, which sorts last)
    for (int j = 0; j < ipt; ++j) {
        const int k = k0 + j;
        keys[k] = k < nb ? pack_key(bs[b0 + k], static_cast<uint32_t>(k)) : 0ull;
    }
    __syncthreads();

    // 2. LSD radix sort, descending = ascending on ~key
    int idx_bits = 0;
    while ((1 << idx_bits) < nb) idx_bits += 4;
    const int npass = idx_bits / 4 + 8;
    for (int ps = 0; ps < npass; ++ps) {
        const int shift = ps < idx_bits / 4 ? 4 * ps : 32 + 4 * (ps - idx_bits / 4);
#pragma unroll
        for (int d = 0; d < kDigits; ++d) cnt[d * kThreads + tid] = 0;
        uint32_t rank[kMaxIpt];
        uint32_t dig[kMaxIpt];
#pragma unroll
        for (int j = 0; j < kMaxIpt; ++j) {
            if (j < ipt) {
                const uint32_t d = static_cast<uint32_t>((~keys[k0 + j]) >> shift) & 15u;
                dig[j] = d;
                rank[j] = cnt[d * kThreads + tid]++;
            }
        }
        __syncthreads();
        // exclusive scan over cnt in (digit, thread) order: 16 consecutive entries per thread
        uint32_t loc[kDigits];
        uint32_t sum = 0;
#pragma unroll
        for (int e = 0; e < kDigits; ++e) {
            loc[e] = cnt[tid * kDigits + e];
            sum += loc[e];
        }
        int tot;
        uint32_t run = static_cast<uint32_t>(block_exclusive_scan<int>(static_cast<int>(sum), shi, &tot));
#pragma unroll
        for (int e = 0; e < kDigits; ++e) {
            const uint32_t c = loc[e];
            cnt[tid * kDigits + e] = run;
            run += c;
        }
        __syncthreads();
#pragma unroll
        for (int j = 0; j < kMaxIpt; ++j)
            if (j < ipt) alt[cnt[dig[j] * kThreads + tid] + rank[j]] = keys[k0 + j];
        __syncthreads();
        uint64_t* t = keys;
        keys = alt;
        alt = t;
    }

    // 3. prefix sums of the sorted scores in fp64 and k*; the threshold uses the last prefix sum
    auto score_of = [&](int k) {
        return static_cast<double>(__uint_as_float(static_cast<uint32_t>(keys[k] >> 32) ^ 0x80000000u));
    };
    double part = 0.0;
    for (int j = 0; j < ipt; ++j)
        if (k0 + j < nb) part += score_of(k0 + j);
    double grand;
    const double before = block_exclusive_scan<double>(part, shd, &grand);
    (void)grand;
    if (k0 <= nb - 1 && nb - 1 < k0 + ipt) {
        double run = before;
        for (int k = k0; k < nb; ++k) run += score_of(k);
        s_total = run;
    }
    __syncthreads();
    const double thr = p * s_total;
    int below = 0;
    double run = before;
    for (int j = 0; j < ipt; ++j) {
        const int k = k0 + j;
        if (k < nb) {
            run += score_of(k);
            below += run < thr;
        }
    }
    int nbelow;
    (void)block_exclusive_scan<int>(below, shi, &nbelow);
    const int ks = min(nb, nbelow + 1);

    // 4. ranked flags by block index, then block and token masks
    for (int j = 0; j < ipt; ++j) {
        const int k = k0 + j;
        if (k < nb) ranked[static_cast<uint32_t>(keys[k])] = k < ks;
    }
    __syncthreads();
    for (int g = tid; g < nb; g += kThreads) {
        const bool forced = (static_cast<int64_t>(g) * G < A) || (static_cast<int64_t>(g + 1) * G > static_cast<int64_t>(N) - n);
        block_keep[b0 + g] = (ranked[g] || forced) ? 1 : 0;
    }
    for (int i = tid; i < N; i += kThreads) {
        const bool keep = ranked[i / G] || i < A || i >= N - n;
        token_keep[c0 + i] = keep ? 1 : 0;
    }
    if (tid == 0) kstar[r] = ks;
}

constexpr int kSmemBytes = 2 * UP_MAX_BLOCKS_PER_REQUEST * 8 + kDigits * kThreads * 4 + UP_MAX_BLOCKS_PER_REQUEST;

__global__ void __launch_bounds__(1024) cu_blocks_kernel(const int32_t* cu, int R, int T, int G, int32_t* cb,
                                                         int32_t* status) {
    __shared__ int sh[32];
    __shared__ int s_bad;
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    if (tid == 0) s_bad = 0;
    __syncthreads();
    for (int r = tid; r < R; r += blockDim.x) {
        const int c0 = cu[r], c1 = cu[r + 1];
        if ((r == 0 && c0 != 0) || c1 < c0 || c1 > T || (r == R - 1 && c1 != T)) s_bad = 1;
    }
    __syncthreads();
    if (s_bad) {
        if (tid == 0) set_status(status, UP_DEV_BAD_CU_SEQLENS);
        return;
    }
    const int per = (R + blockDim.x - 1) / blockDim.x;
    const int r0 = min(R, tid * per), r1 = min(R, r0 + per);
    int local = 0;
    for (int r = r0; r < r1; ++r) local += (cu[r + 1] - cu[r] + G - 1) / G;
    int x = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) sh[w] = x;
    __syncthreads();
    if (w == 0) {
        int s = sh[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o) s += y;
        }
        sh[lane] = s;
    }
    __syncthreads();
    int off = (w > 0 ? sh[w - 1] : 0) + x - local;
    if (tid == 0) cb[0] = 0;
    for (int r = r0; r < r1; ++r) {
        off += (cu[r + 1] - cu[r] + G - 1) / G;
        cb[r + 1] = off;
    }
}

}  // namespace select
}  // namespace up

using namespace up;

extern "C" up_status up_make_cu_blocks(const int32_t* cu_seqlens, int R, int64_t T, int G, int32_t* cu_blocks,
                                       int32_t* dev_status, void* stream) {
    if (!cu_seqlens || !cu_blocks || !dev_status) return UP_ERR_ARG;
    if (R <= 0 || T < 0 || T >= (int64_t(1) << 31) || G <= 0) return UP_ERR_ARG;
    select::cu_blocks_kernel<<<1, 1024, 0, static_cast<cudaStream_t>(stream)>>>(cu_seqlens, R, static_cast<int>(T),
                                                                                G, cu_blocks, dev_status);
    count_launch();
    return check_launch();
}

extern "C" up_status up_select_topp(const float* block_scores, const int32_t* cu_blocks, const int32_t* cu_seqlens,
                                    int R, int64_t T, int64_t nb_cap, int G, int n, int A, double p,
                                    uint8_t* block_keep, uint8_t* token_keep, int32_t* kstar, int32_t* dev_status,
                                    void* stream) {
    if (!block_scores || !cu_blocks || !cu_seqlens || !block_keep || !token_keep || !kstar || !dev_status)
        return UP_ERR_ARG;
    if (R <= 0 || T < 0 || T >= (int64_t(1) << 31) || nb_cap < 0 || G <= 0 || n < 1 || A < 0) return UP_ERR_ARG;
    if (!(p > 0.0) || !(p <= 1.0)) return UP_ERR_ARG;
    static int attr_done[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return UP_ERR_CUDA;
    if (dev < 64 && !attr_done[dev]) {
        if (cudaFuncSetAttribute(select::select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 select::kSmemBytes) != cudaSuccess)
            return UP_ERR_CUDA;
        attr_done[dev] = 1;
    }
    select::select_kernel<<<R, select::kThreads, select::kSmemBytes, static_cast<cudaStream_t>(stream)>>>(
        block_scores, cu_blocks, cu_seqlens, R, static_cast<int>(T), nb_cap, G, n, A, p, block_keep, token_keep,
        kstar, dev_status);
    count_launch();
    return check_launch();
}
