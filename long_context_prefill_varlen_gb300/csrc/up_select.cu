// up_select_topp and up_make_cu_blocks: top-p block selection of UniPrefill ("UniPrefill:
// Universal Long-Context Prefill Acceleration via Block-wise Dynamic Sparsification",
// arXiv 2605.06221, section 3.3 Eq. 5 with the forced sink/window tokens, and the top-p kernel of
// section 3.5 with the packed sort key of Eq. 14).
//
// One CTA per request, no CPU round trip.  Requests of at most UP_MAX_BLOCKS_PER_REQUEST blocks keep
// everything in shared memory; longer ones run the same passes over their keys in the caller's
// workspace (select_large below):
//   1. key_g = (phi(b_g) << 32) | g for the request's blocks (phi(x) = bits(x) ^ 0x80000000 for
//      x >= 0; scores are non-negative sums of probabilities, so the sign bit decides phi).
//   2. LSD radix sort of the 64-bit keys, descending, 8-bit digits, stable.  The keys are laid out
//      in descending order of g before the first pass, which is exactly the order the passes over
//      the low (index) word would produce, so only the four passes over the high word run.  The
//      result is the descending order of the packed 64-bit keys.
//   3. inclusive prefix sum of the sorted scores in fp64 (fixed tree), k* = 1 + #{k : cum_k < p*total}.
//   4. ranked flags by block index, then the byte masks: block(i) ranked, or i < A, or i >= N - n.
#include <stdint.h>

#include "up_internal.cuh"

namespace up {
namespace select {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxIpt = UP_MAX_BLOCKS_PER_REQUEST / kThreads;   // 16 keys per thread
constexpr int kRadix = 256;

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

// Token mask of one request: byte i is ranked(i >> log2 G) or a sink (i < A) or a window token
// (i >= N - n); the aligned interior is written 16 bytes per store (token_keep is 16-byte aligned), the
// unaligned head and tail byte by byte.
template <typename RankedFn>
__device__ __forceinline__ void write_token_mask(uint8_t* token_keep, int T, int c0, int N, int G, int A, int n,
                                                 RankedFn ranked, int32_t* status) {
    const int tid = threadIdx.x;
    const int gshift = __ffs(G) - 1;
    auto keep_byte = [&](int i) -> uint32_t { return (ranked(i >> gshift) || i < A || i >= N - n) ? 1u : 0u; };
    const int64_t a0 = c0, a1 = (int64_t)c0 + N;
    const int64_t v0 = min((a0 + 15) & ~int64_t(15), a1), v1 = max(a1 & ~int64_t(15), v0);
    for (int64_t t = a0 + tid; t < v0; t += kThreads)
        if (UP_IN(t, T, status)) token_keep[t] = static_cast<uint8_t>(keep_byte(static_cast<int>(t - a0)));
    for (int64_t t = v1 + tid; t < a1; t += kThreads)
        if (UP_IN(t, T, status)) token_keep[t] = static_cast<uint8_t>(keep_byte(static_cast<int>(t - a0)));
    // with the request start 16-byte aligned and G >= 16, a 16-byte group lies in one block; clear
    // of the sinks and the window it is that block's flag repeated
    const bool whole = G >= 16 && v0 == a0;
    for (int64_t t = v0 + 16 * (int64_t)tid; t < v1; t += 16 * (int64_t)kThreads) {
        if (!UP_IN(t + 15, T, status)) continue;
        const int i0 = static_cast<int>(t - a0);
        if (whole && i0 >= A && i0 + 15 < N - n) {
            const uint32_t b = ranked(i0 >> gshift) ? 0x01010101u : 0u;
            *reinterpret_cast<uint4*>(token_keep + t) = make_uint4(b, b, b, b);
            continue;
        }
        uint32_t w[4];
#pragma unroll
        for (int q = 0; q < 4; ++q)
            w[q] = keep_byte(i0 + 4 * q) | (keep_byte(i0 + 4 * q + 1) << 8) | (keep_byte(i0 + 4 * q + 2) << 16) |
                   (keep_byte(i0 + 4 * q + 3) << 24);
        *reinterpret_cast<uint4*>(token_keep + t) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// Requests of more than UP_MAX_BLOCKS_PER_REQUEST blocks: the keys go through the caller's workspace
// (two arrays of nb_cap words, this request at offset b0 of each).  The same four stable 8-bit passes
// over the score word, in tiles of kThreads * kMaxIpt keys: a digit count over the whole request gives
// each digit's first destination, then the tiles are ranked in (digit, warp, round, lane) order as above
// and scattered in tile order, so the passes stay stable.  The fp64 prefix sums then run tile by tile
// with a carry; the total is the last prefix sum, computed in the same order.  Ranked flags go to
// block_keep, from which the token mask is written; the forced blocks are set last.
__device__ __noinline__ void select_large(const float* __restrict__ bs, int b0, int nb, int64_t nb_cap, int c0, int N,
                                          int G, int n, int A, double p, uint64_t* ws_keys, uint8_t* block_keep,
                                          uint8_t* token_keep, int32_t* kstar, int r, int T, uint8_t* sm,
                                          double* shd, int* shi, double* s_total, int* s_below, int32_t* status) {
    constexpr int kTileKeys = kThreads * kMaxIpt;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint64_t* src = ws_keys + b0;
    uint64_t* dst = ws_keys + nb_cap + b0;
    uint32_t* hist = reinterpret_cast<uint32_t*>(sm);                   // [kRadix digits][kWarps]
    uint32_t* dbase = hist + kRadix * kWarps;                           // [kRadix] next destination of a digit
    for (int k = tid; k < nb; k += kThreads) {                          // position k holds block nb - 1 - k
        const int g = nb - 1 - k;
        if (UP_IN(b0 + k, nb_cap, status) && UP_IN(b0 + g, nb_cap, status))
            src[k] = pack_key(bs[b0 + g], static_cast<uint32_t>(g));
    }
    __syncthreads();
    const uint32_t lt_mask = (1u << lane) - 1u;
    for (int ps = 0; ps < 4; ++ps) {
        const int shift = 32 + 8 * ps;
        for (int i = tid; i < kRadix; i += kThreads) dbase[i] = 0;
        __syncthreads();
        for (int k = tid; k < nb; k += kThreads) atomicAdd(&dbase[static_cast<uint32_t>((~src[k]) >> shift) & 0xFFu], 1u);
        __syncthreads();
        {
            int tot;
            const int ex = block_exclusive_scan<int>(tid < kRadix ? static_cast<int>(dbase[tid]) : 0, shi, &tot);
            if (tid < kRadix) dbase[tid] = static_cast<uint32_t>(ex);
        }
        __syncthreads();
        for (int t0 = 0; t0 < nb; t0 += kTileKeys) {
            for (int i = tid; i < kRadix * kWarps; i += kThreads) hist[i] = 0;
            __syncthreads();
            uint32_t rank[kMaxIpt], dig[kMaxIpt];
            const int base_k = t0 + warp * 32 * kMaxIpt + lane;
#pragma unroll
            for (int j = 0; j < kMaxIpt; ++j) {
                const int k = base_k + 32 * j;
                const uint32_t d = k < nb ? static_cast<uint32_t>((~src[k]) >> shift) & 0xFFu : 0x100u;   // 0x100: none
                const uint32_t peers = __match_any_sync(0xffffffffu, d);
                const uint32_t before = d < 0x100u ? hist[d * kWarps + warp] : 0u;
                __syncwarp();
                if (d < 0x100u && (peers & lt_mask) == 0) hist[d * kWarps + warp] = before + __popc(peers);
                __syncwarp();
                dig[j] = d;
                rank[j] = before + __popc(peers & lt_mask);
            }
            __syncthreads();
            if (tid < kRadix) {                 // digit tid: its warps' first destinations in this tile
                uint32_t run = dbase[tid];
                for (int w2 = 0; w2 < kWarps; ++w2) {
                    const uint32_t c = hist[tid * kWarps + w2];
                    hist[tid * kWarps + w2] = run;
                    run += c;
                }
                dbase[tid] = run;
            }
            __syncthreads();
#pragma unroll
            for (int j = 0; j < kMaxIpt; ++j)
                if (dig[j] < 0x100u && UP_IN(hist[dig[j] * kWarps + warp] + rank[j], nb, status))
                    dst[hist[dig[j] * kWarps + warp] + rank[j]] = src[base_k + 32 * j];
            __syncthreads();
        }
        uint64_t* t = src;
        src = dst;
        dst = t;
    }
    // the sorted keys are in src (an even number of passes).  Prefix sums: thread tid of a tile sums the
    // tile's positions tid * kMaxIpt .. + kMaxIpt - 1 in order, a block scan orders the threads, and the
    // tiles are chained by a carry that every thread computes identically.
    auto score_of = [&](int k) {
        return static_cast<double>(__uint_as_float(static_cast<uint32_t>(src[k] >> 32) ^ 0x80000000u));
    };
    auto sweep = [&](bool count, double thr) {
        double carry = 0.0;
        int below = 0;
        for (int t0 = 0; t0 < nb; t0 += kTileKeys) {
            const int k0 = t0 + tid * kMaxIpt;
            double part = 0.0;
            for (int j = 0; j < kMaxIpt; ++j)
                if (k0 + j < nb) part += score_of(k0 + j);
            double tot;
            const double before = block_exclusive_scan<double>(part, shd, &tot);
            if (count || (k0 <= nb - 1 && nb - 1 < k0 + kMaxIpt)) {
                double run = carry + before;
                for (int j = 0; j < kMaxIpt; ++j) {
                    if (k0 + j < nb) {
                        run += score_of(k0 + j);
                        below += run < thr;
                    }
                }
                if (!count && k0 <= nb - 1 && nb - 1 < k0 + kMaxIpt) *s_total = run;
            }
            carry += tot;
        }
        return below;
    };
    sweep(false, 0.0);
    __syncthreads();
    const double thr = p * *s_total;
    const int below = sweep(true, thr);
    if (tid == 0) *s_below = 0;
    __syncthreads();
    if (below) atomicAdd(s_below, below);
    __syncthreads();
    const int ks = min(nb, *s_below + 1);
    for (int k = tid; k < nb; k += kThreads) {
        const uint32_t g = static_cast<uint32_t>(src[k]);
        if (UP_IN(g, nb, status)) block_keep[b0 + g] = k < ks ? 1 : 0;
    }
    __syncthreads();
    write_token_mask(token_keep, T, c0, N, G, A, n, [&](int g) { return block_keep[b0 + g] != 0; }, status);
    __syncthreads();
    for (int g = tid; g < nb; g += kThreads) {
        const bool forced = (static_cast<int64_t>(g) * G < A) || (static_cast<int64_t>(g + 1) * G > static_cast<int64_t>(N) - n);
        if (forced && UP_IN(b0 + g, nb_cap, status)) block_keep[b0 + g] = 1;
    }
    if (tid == 0) kstar[r] = ks;
}

__global__ void __launch_bounds__(kThreads) select_kernel(const float* __restrict__ bs, const int32_t* __restrict__ cb,
                                                          const int32_t* __restrict__ cu, int R, int T, int64_t nb_cap,
                                                          int G, int n, int A, double p, uint8_t* block_keep,
                                                          uint8_t* token_keep, int32_t* kstar, uint64_t* ws_keys,
                                                          int32_t* status) {
    pdl_wait();
    pdl_trigger();
    extern __shared__ __align__(16) uint8_t sm[];
    uint64_t* keys = reinterpret_cast<uint64_t*>(sm);                              // [8192]
    uint64_t* alt = keys + UP_MAX_BLOCKS_PER_REQUEST;                              // [8192]
    uint32_t* hist = reinterpret_cast<uint32_t*>(alt + UP_MAX_BLOCKS_PER_REQUEST); // [256 digits][16 warps]
    uint8_t* ranked = reinterpret_cast<uint8_t*>(hist + kRadix * kWarps);          // [8192]
    __shared__ double shd[65];
    __shared__ int shi[65];
    __shared__ double s_total;
    __shared__ int s_bad;
    __shared__ int s_below;

    const int r = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int c0 = cu[r], c1 = cu[r + 1];
    const int N = c1 - c0;
    const int nb = N > 0 ? (N + G - 1) / G : 0;
    if (tid == 0) {
        int bad = 0;
        if ((r == 0 && c0 != 0) || c1 < c0 || c1 > T || (r == R - 1 && c1 != T)) bad = UP_DEV_BAD_CU_SEQLENS;
        else if ((r == 0 && cb[0] != 0) || cb[r + 1] - cb[r] != nb || (int64_t)cb[r + 1] > nb_cap) bad = UP_DEV_BAD_CU_BLOCKS;
        else if (nb > UP_MAX_BLOCKS_PER_REQUEST && ws_keys == nullptr) bad = UP_DEV_TOO_MANY_BLOCKS;
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
    if (nb > UP_MAX_BLOCKS_PER_REQUEST) {
        select_large(bs, b0, nb, nb_cap, c0, N, G, n, A, p, ws_keys, block_keep, token_keep, kstar, r, T, sm, shd,
                     shi, &s_total, &s_below, status);
        return;
    }
    const int ipt = (nb + kThreads - 1) / kThreads;      // keys per thread
    const int npad = ipt * kThreads;

    // 1. packed keys, position k holds block g = nb-1-k (padding slots get key 0, which sorts last)
    for (int k = tid; k < npad; k += kThreads) {
        const int g = nb - 1 - k;
        keys[k] = g >= 0 && UP_IN(b0 + g, nb_cap, status) ? pack_key(bs[b0 + g], static_cast<uint32_t>(g)) : 0ull;
    }
    __syncthreads();

    if (ipt == 1) {
        // 2a. at most kThreads blocks: a bitonic network over the whole 64-bit keys, one key per thread
        //     (padding keys are 0 and sort last).  The keys are distinct (the block index is the low
        //     word), so the descending order is the one the radix passes below produce.  Partners in
        //     the same warp are exchanged by shuffle, the others through two alternating shared
        //     buffers (one barrier per such step).
        uint64_t v = keys[tid];
        int par = 0;
        for (int k = 2; k <= kThreads; k <<= 1) {
            for (int j = k >> 1; j > 0; j >>= 1) {
                uint64_t o;
                if (j < 32) {
                    o = __shfl_xor_sync(0xffffffffu, v, j);
                } else {
                    uint64_t* xb = alt + par * kThreads;
                    xb[tid] = v;
                    __syncthreads();
                    o = xb[tid ^ j];
                    par ^= 1;
                }
                const bool lower = (tid & j) == 0, desc = (tid & k) == 0;
                v = (lower == desc) ? (v > o ? v : o) : (v < o ? v : o);
            }
        }
        keys[tid] = v;
        __syncthreads();
    } else {
        // 2. four stable passes over the high word, ascending on ~key (= descending on key).  Warp w owns
        //    positions [w*32*ipt, (w+1)*32*ipt), visited round by round (32 consecutive keys per round), so
        //    (digit, warp, round, lane) order equals (digit, position) order: the passes are stable.
        const uint32_t lt_mask = (1u << lane) - 1u;
        for (int ps = 0; ps < 4; ++ps) {
            const int shift = 32 + 8 * ps;
            for (int i = tid; i < kRadix * kWarps; i += kThreads) hist[i] = 0;
            __syncthreads();
            uint32_t rank[kMaxIpt];
            uint32_t dig[kMaxIpt];
            const int base_k = warp * 32 * ipt + lane;
#pragma unroll
            for (int j = 0; j < kMaxIpt; ++j) {
                if (j < ipt) {
                    const uint32_t d = static_cast<uint32_t>((~keys[base_k + 32 * j]) >> shift) & 0xFFu;
                    const uint32_t peers = __match_any_sync(0xffffffffu, d);
                    const uint32_t before = hist[d * kWarps + warp];
                    __syncwarp();
                    if ((peers & lt_mask) == 0) hist[d * kWarps + warp] = before + __popc(peers);
                    __syncwarp();
                    dig[j] = d;
                    rank[j] = before + __popc(peers & lt_mask);
                }
            }
            __syncthreads();
            // exclusive scan of hist in (digit, warp) order: 8 consecutive entries per thread
            uint32_t loc[8];
            uint32_t sum = 0;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                loc[e] = hist[tid * 8 + e];
                sum += loc[e];
            }
            int tot;
            uint32_t run = static_cast<uint32_t>(block_exclusive_scan<int>(static_cast<int>(sum), shi, &tot));
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const uint32_t c = loc[e];
                hist[tid * 8 + e] = run;
                run += c;
            }
            __syncthreads();
#pragma unroll
            for (int j = 0; j < kMaxIpt; ++j)
                if (j < ipt) alt[hist[dig[j] * kWarps + warp] + rank[j]] = keys[base_k + 32 * j];
            __syncthreads();
            uint64_t* t = keys;
            keys = alt;
            alt = t;
        }
    }
    const int k0 = tid * ipt;      // from here on each thread owns a contiguous run of sorted positions

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
    if (tid == 0) s_below = 0;                     // #{k : cum_k < thr}: an integer count, any order
    __syncthreads();
    if (below) atomicAdd(&s_below, below);
    __syncthreads();
    const int ks = min(nb, s_below + 1);

    // 4. ranked flags by block index, then block and token masks
    for (int j = 0; j < ipt; ++j) {
        const int k = k0 + j;
        if (k < nb && UP_IN(static_cast<uint32_t>(keys[k]), UP_MAX_BLOCKS_PER_REQUEST, status))
            ranked[static_cast<uint32_t>(keys[k])] = k < ks;
    }
    __syncthreads();
    for (int g = tid; g < nb; g += kThreads) {
        const bool forced = (static_cast<int64_t>(g) * G < A) || (static_cast<int64_t>(g + 1) * G > static_cast<int64_t>(N) - n);
        if (UP_IN(b0 + g, nb_cap, status)) block_keep[b0 + g] = (ranked[g] || forced) ? 1 : 0;
    }
    write_token_mask(token_keep, T, c0, N, G, A, n, [&](int g) { return ranked[g] != 0; }, status);
    if (tid == 0) kstar[r] = ks;
}

constexpr int kSmemBytes = 2 * UP_MAX_BLOCKS_PER_REQUEST * 8 + kRadix * kWarps * 4 + UP_MAX_BLOCKS_PER_REQUEST;

__global__ void __launch_bounds__(1024) cu_blocks_kernel(const int32_t* cu, int R, int T, int G, int32_t* cb,
                                                         int32_t* status) {
    pdl_wait();
    pdl_trigger();
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
    launch_pdl(select::cu_blocks_kernel, dim3(1), dim3(1024), 0, static_cast<cudaStream_t>(stream),
        cu_seqlens, R, static_cast<int>(T), G, cu_blocks, dev_status);
    count_launch();
    return check_launch();
}

extern "C" size_t up_select_workspace_bytes(int64_t nb_cap) {
    if (nb_cap < 0) return 0;
    return align_up(sizeof(uint64_t) * 2 * static_cast<size_t>(nb_cap), 256);
}

extern "C" up_status up_select_topp(const float* block_scores, const int32_t* cu_blocks, const int32_t* cu_seqlens,
                                    int R, int64_t T, int64_t nb_cap, int G, int n, int A, double p,
                                    uint8_t* block_keep, uint8_t* token_keep, int32_t* kstar, void* ws,
                                    size_t ws_bytes, int32_t* dev_status, void* stream) {
    // token_keep may be NULL for a batch without tokens (T = 0)
    if (!block_scores || !cu_blocks || !cu_seqlens || !block_keep || (T > 0 && !token_keep) || !kstar || !dev_status)
        return UP_ERR_ARG;
    if (R <= 0 || T < 0 || T >= (int64_t(1) << 31) || nb_cap < 0 || G <= 0 || n < 1 || A < 0) return UP_ERR_ARG;
    if (!(p > 0.0) || !(p <= 1.0)) return UP_ERR_ARG;
    if (G & (G - 1)) return UP_ERR_SHAPE;          // block size must be a power of two
    if (T > 0 && !aligned16(token_keep)) return UP_ERR_SHAPE;   // the mask is written 16 bytes per store
    if (ws != nullptr && (!aligned16(ws) || ws_bytes < up_select_workspace_bytes(nb_cap))) return UP_ERR_WORKSPACE;
    static int attr_done[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return UP_ERR_CUDA;
    if (dev < 64 && !attr_done[dev]) {
        if (cudaFuncSetAttribute(select::select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 select::kSmemBytes) != cudaSuccess)
            return UP_ERR_CUDA;
        attr_done[dev] = 1;
    }
    launch_pdl(select::select_kernel, dim3(R), dim3(select::kThreads), select::kSmemBytes,
        static_cast<cudaStream_t>(stream), block_scores, cu_blocks, cu_seqlens, R, static_cast<int>(T), nb_cap, G, n, A, p, block_keep, token_keep,
        kstar, static_cast<uint64_t*>(ws), dev_status);
    count_launch();
    return check_launch();
}
