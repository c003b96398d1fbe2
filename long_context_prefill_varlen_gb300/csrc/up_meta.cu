// Metadata for downstream layers and decode (section 3.5 of "UniPrefill: Universal Long-Context
// Prefill Acceleration via Block-wise Dynamic Sparsification", arXiv 2605.06221):
//   up_slot_mapping  Eq. 16, KV slot ids of a (compacted) token stream from a layer's block table
//   up_seqused       Eq. 17, the KV length each layer saw during prefill, from the drop history
// plus the status word reader, status strings and the launch counter.
#include <atomic>
#include <mutex>

#include <algorithm>

#include "up_internal.cuh"

namespace up {

static std::atomic<uint64_t> g_launches{0};
void count_launch(int n) { g_launches.fetch_add(static_cast<uint64_t>(n), std::memory_order_relaxed); }

int num_sms() {
    static int cache[64] = {0};
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    std::lock_guard<std::mutex> lk(mu);
    if (dev >= 0 && dev < 64 && cache[dev] > 0) return cache[dev];
    int v = 1;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 1;
    if (dev >= 0 && dev < 64) cache[dev] = v;
    return v;
}

up_status check_launch() { return cudaGetLastError() == cudaSuccess ? UP_OK : UP_ERR_CUDA; }

namespace meta {

__global__ void slot_kernel(const int64_t* __restrict__ pos, const int32_t* __restrict__ cu, int R, int64_t T_upper,
                            const int32_t* __restrict__ num_tokens, const int32_t* __restrict__ table, int max_blocks,
                            int B, int64_t* slots, int32_t* status) {
    pdl_wait();
    pdl_trigger();
    int64_t n = T_upper;
    if (num_tokens) {
        const int c = *num_tokens;
        if (c < 0 || c > T_upper) {
            if (blockIdx.x == 0 && threadIdx.x == 0) set_status(status, UP_DEV_BAD_TOKEN_COUNT);
            return;
        }
        n = c;
    }
    for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < n; t += (int64_t)gridDim.x * blockDim.x) {
        int lo = 0, hi = R;   // request r with cu[r] <= t < cu[r+1]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (cu[mid] <= t) lo = mid; else hi = mid;
        }
        if (!UP_IN(t, T_upper, status)) continue;
        const int64_t p = pos[t];
        const int64_t blk = p >= 0 ? p / B : -1;
        if (p < 0 || blk >= max_blocks || t >= cu[R]) {
            slots[t] = -1;
            set_status(status, UP_DEV_BAD_POSITION);
        } else {
            const int64_t e = (int64_t)lo * max_blocks + blk;
            slots[t] = UP_IN(e, (int64_t)R * max_blocks, status) ? static_cast<int64_t>(table[e]) * B + (p % B) : -1;
        }
    }
}

__global__ void seqused_kernel(const int32_t* __restrict__ kept_len, const uint8_t* __restrict__ drop_layer, int L,
                               int R, int layer, const int32_t* __restrict__ orig_len,
                               const int32_t* __restrict__ kv_len, int32_t* seqused) {
    pdl_wait();
    pdl_trigger();
    __shared__ int s_prev;
    if (threadIdx.x == 0) {
        int prev = -1;
        for (int l = 0; l < layer && l < L; ++l)
            if (drop_layer[l]) prev = l;
        s_prev = prev;
    }
    __syncthreads();
    const int prev = s_prev;
    for (int r = blockIdx.x * blockDim.x + threadIdx.x; r < R; r += gridDim.x * blockDim.x) {
        // up_seqused has no status word: an index outside kept_len is skipped, not reported
        if (prev >= 0 && !UP_IN((int64_t)prev * R + r, (int64_t)L * R, nullptr)) continue;
        const int base = prev >= 0 ? kept_len[(int64_t)prev * R + r] : orig_len[r];
        seqused[r] = base + (kv_len[r] - orig_len[r]);
    }
}

}  // namespace meta
}  // namespace up

using namespace up;

extern "C" up_status up_slot_mapping(const int64_t* positions, const int32_t* cu_seqlens, int R, int64_t T_upper,
                                     const int32_t* num_tokens, const int32_t* block_table, int max_blocks, int B,
                                     int64_t* slots, int32_t* dev_status, void* stream) {
    if (!cu_seqlens || !block_table || !dev_status) return UP_ERR_ARG;
    if (R <= 0 || T_upper < 0 || max_blocks <= 0 || B <= 0) return UP_ERR_ARG;
    if (T_upper == 0) return UP_OK;        // no tokens: positions and slots may be empty (NULL)
    if (!positions || !slots) return UP_ERR_ARG;
    const int grid = static_cast<int>(std::min<int64_t>(cdiv(T_upper, 256), 8 * num_sms()));
    launch_pdl(meta::slot_kernel, dim3(grid), dim3(256), 0, static_cast<cudaStream_t>(stream),
        positions, cu_seqlens, R, T_upper, num_tokens, block_table, max_blocks, B, slots, dev_status);
    count_launch();
    return check_launch();
}

extern "C" up_status up_seqused(const int32_t* kept_len, const uint8_t* drop_layer, int L, int R, int layer,
                                const int32_t* orig_len, const int32_t* kv_len, int32_t* seqused, void* stream) {
    if (!kept_len || !drop_layer || !orig_len || !kv_len || !seqused) return UP_ERR_ARG;
    if (L <= 0 || R <= 0 || layer < 0 || layer >= L) return UP_ERR_ARG;
    const int grid = static_cast<int>(std::min<int64_t>(cdiv(R, 256), 4 * num_sms()));
    launch_pdl(meta::seqused_kernel, dim3(grid), dim3(256), 0, static_cast<cudaStream_t>(stream),
        kept_len, drop_layer, L, R, layer, orig_len, kv_len, seqused);
    count_launch();
    return check_launch();
}

extern "C" up_status up_read_status(const int32_t* dev_status, int32_t* host_out, void* stream) {
    if (!dev_status || !host_out) return UP_ERR_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(host_out, dev_status, sizeof(int32_t), cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return UP_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return UP_ERR_CUDA;
    return *host_out == 0 ? UP_OK : UP_ERR_DEVICE;
}

extern "C" const char* up_status_string(int code, int device) {
    if (device) {
        switch (code) {
            case UP_DEV_OK: return "ok";
            case UP_DEV_BAD_CU_SEQLENS: return "cu_seqlens is not a non-decreasing 0..T sequence";
            case UP_DEV_BAD_CU_BLOCKS: return "cu_blocks does not match ceil(N_r/G) or exceeds nb_cap";
            case UP_DEV_TOO_MANY_BLOCKS: return "a request has more blocks than UP_MAX_BLOCKS_PER_REQUEST";
            case UP_DEV_WAIT_TIMEOUT: return "a pipeline wait inside a kernel exceeded its time bound";
            case UP_DEV_BAD_POSITION: return "a position lies outside its block-table row";
            case UP_DEV_BAD_TOKEN_COUNT: return "num_actual_tokens lies outside [0, T_upper]";
            case UP_DEV_BOUNDS: return "an index lies outside its array (bounds-checked build)";
            default: return "unknown device status";
        }
    }
    switch (code) {
        case UP_OK: return "UP_OK";
        case UP_ERR_ARG: return "UP_ERR_ARG: null pointer or scalar out of range";
        case UP_ERR_SHAPE: return "UP_ERR_SHAPE: unsupported geometry or alignment";
        case UP_ERR_WORKSPACE: return "UP_ERR_WORKSPACE: workspace too small";
        case UP_ERR_CUDA: return "UP_ERR_CUDA: CUDA runtime or launch failure";
        case UP_ERR_DEVICE: return "UP_ERR_DEVICE: a kernel reported an error in dev_status";
        default: return "unknown status";
    }
}

extern "C" uint64_t up_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

extern "C" int up_abi_version(void) { return 2; }

extern "C" int up_debug_bounds(void) {
#ifdef UP_DEBUG_BOUNDS
    return 1;
#else
    return 0;
#endif
}

extern "C" size_t up_workspace_bytes(int R, int64_t T, int Hq, int Hkv, int dk, int G, int n, int64_t nb_cap) {
    const size_t a = up_score_workspace_bytes(R, T, Hq, Hkv, dk, G, n, nb_cap, 1);
    const size_t b = up_compact_workspace_bytes(R, T);
    const size_t c = up_select_workspace_bytes(nb_cap);
    if (a == 0 || b == 0) return 0;
    const size_t ab = a > b ? a : b;
    return ab > c ? ab : c;
}
