// up_compact and up_scatter_back: the token-stream side of UniPrefill ("UniPrefill: Universal
// Long-Context Prefill Acceleration via Block-wise Dynamic Sparsification", arXiv 2605.06221):
// compaction of the kept tokens with the patched query_start_loc / seq_lens / num_actual_tokens
// and the drop-history record (section 3.5, "vLLM scheduler integration"), and the end-of-block
// carry-forward of Eq. 8 (section 3.4).
//
// Compaction is three launches, none of which waits on another CTA (two for streams of at most
// kScanCountTiles tiles, whose scan kernel counts the tiles itself, and one for streams of at most
// kSelfScanTiles tiles, whose gather CTAs each count and scan the tiles; for longer streams that
// repeated read of the mask by every CTA concentrated on a few L2 slices and slowed the step):
//   count   per 1024-token tile, the number of kept tokens (16-byte loads of the byte mask)
//   scan    one CTA: tile offsets, and per request prefix(cu[r]) = kept tokens before cu[r]
//           -> new_cu_seqlens, new_seq_lens, num_actual_tokens, kept_len[layer], drop_layer[layer]
//   gather  persistent CTAs over (tile, part) items, parts chosen so that there are about 32 items per
//           resident CTA: a scan of the tile's flags gives each kept token its place; part 0 writes
//           kept_index, out_positions and out_slots, every part copies its share of the kept hidden
//           rows with 16-byte vectors, one warp per row (HBM bound: 2 * T' * hdim * 2 bytes)
// Scatter-back is the row copy in the other direction: residual[kept_index[k]] = new_states[k].
#include <stdint.h>

#include <algorithm>
#include <mutex>

#include "up_internal.cuh"

namespace up {
namespace compact {

constexpr int kTile = 1024;          // tokens per tile
constexpr int kTileThreads = 64;     // 16 flags per thread
constexpr int kRowThreads = 512;
constexpr int kRowUnroll = 8;
constexpr int kGatherThreads = 256;
constexpr int kMaxParts = 64;          // work items sharing one tile's row copies
constexpr int kItemsPerCta = 32;       // gather work items per resident CTA (see launch_gather)
constexpr int kScanCountTiles = 64;    // up to this many tiles the scan kernel counts them itself
constexpr int kSelfScanTiles = 8;      // up to this many tiles the gather scans the stream itself

struct Layout {
    size_t tile_cnt, tile_off, total;
};

static Layout layout(int64_t T) {
    Layout L{};
    const int64_t tiles = cdiv(T, kTile) + 1;
    L.tile_cnt = 0;
    L.tile_off = align_up(sizeof(int) * tiles, 256);
    L.total = L.tile_off + align_up(sizeof(int) * tiles, 256);
    return L;
}

__device__ __forceinline__ int count_nonzero_bytes(uint4 v) {
    // number of non-zero bytes in 16 flag bytes
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    int c = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t x = w[i];
        const uint32_t nz = ((x & 0x7F7F7F7Fu) + 0x7F7F7F7Fu | x) & 0x80808080u;   // high bit set where byte != 0
        c += __popc(nz);
    }
    return c;
}

__device__ __forceinline__ uint4 load_flags16(const uint8_t* f, int64_t t0, int64_t T) {
    if (t0 + 16 <= T) return *reinterpret_cast<const uint4*>(f + t0);
    uint8_t b[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) b[i] = (t0 + i < T) ? f[t0 + i] : 0;
    uint4 v;
    v.x = b[0] | (b[1] << 8) | (b[2] << 16) | ((uint32_t)b[3] << 24);
    v.y = b[4] | (b[5] << 8) | (b[6] << 16) | ((uint32_t)b[7] << 24);
    v.z = b[8] | (b[9] << 8) | (b[10] << 16) | ((uint32_t)b[11] << 24);
    v.w = b[12] | (b[13] << 8) | (b[14] << 16) | ((uint32_t)b[15] << 24);
    return v;
}

__device__ __forceinline__ int block_reduce(int v, int* sh) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) sh[w] = v;
    __syncthreads();
    int t = 0;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kTileThreads / 32; ++i) t += sh[i];
        sh[8] = t;
    }
    __syncthreads();
    t = sh[8];
    __syncthreads();
    return t;
}

__global__ void __launch_bounds__(kTileThreads) count_kernel(const uint8_t* __restrict__ keep, int T, int* tile_cnt,
                                                              int tiles, int32_t* status) {
    pdl_wait();
    pdl_trigger();
    __shared__ int sh[9];
    const int64_t t0 = (int64_t)blockIdx.x * kTile + threadIdx.x * 16;
    const int c = t0 < T ? count_nonzero_bytes(load_flags16(keep, t0, T)) : 0;
    const int tot = block_reduce(c, sh);
    if (threadIdx.x == 0 && UP_IN(blockIdx.x, tiles, status)) tile_cnt[blockIdx.x] = tot;
}

// Whether cu_seqlens is a non-decreasing 0..T sequence (all threads of the CTA take part; sh_bad is
// a shared flag).
__device__ __forceinline__ bool cu_valid(const int32_t* __restrict__ cu, int R, int T, int* sh_bad) {
    if (threadIdx.x == 0) *sh_bad = 0;
    __syncthreads();
    for (int r = threadIdx.x; r < R; r += blockDim.x) {
        const int c0 = cu[r], c1 = cu[r + 1];
        if ((r == 0 && c0 != 0) || c1 < c0 || c1 > T || (r == R - 1 && c1 != T)) *sh_bad = 1;
    }
    __syncthreads();
    return *sh_bad == 0;
}

// The per-request side of the compaction, from the tile offsets (off[i] = kept tokens before tile i,
// total = kept tokens of the stream): kept tokens before each request boundary (one warp per
// boundary; the boundary's partial tile is counted flag by flag) -> new_cu_seqlens, new_seq_lens,
// num_actual_tokens and the drop history.  Called by every thread of one CTA, cu_seqlens valid.
__device__ void request_metadata(const uint8_t* __restrict__ keep, const int32_t* __restrict__ cu, int R, int T,
                                 int tiles, const int* off, int total, int32_t* new_cu, int32_t* new_len,
                                 int32_t* num_actual, int32_t* kept_len, uint8_t* drop_layer, int L, int layer,
                                 int32_t* status) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
    for (int r = w; r <= R; r += nw) {
        const int x0 = cu[r];
        const int tile = x0 / kTile;
        int c = 0;
        for (int t = tile * kTile + lane; t < x0; t += 32) c += (UP_IN(t, T, status) ? keep[t] : 0) != 0;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
        if (lane == 0 && UP_IN(r, R + 1, status)) new_cu[r] = (tile < tiles ? off[tile] : total) + c;
    }
    __syncthreads();
    for (int r = threadIdx.x; r < R; r += blockDim.x) {
        const int len = new_cu[r + 1] - new_cu[r];
        new_len[r] = len;
        if (kept_len && UP_IN((int64_t)layer * R + r, (int64_t)L * R, status)) kept_len[(int64_t)layer * R + r] = len;
    }
    if (threadIdx.x == 0) {
        *num_actual = new_cu[R];
        if (drop_layer && UP_IN(layer, L, status)) drop_layer[layer] = 1;
    }
}

// Streams of more than kSelfScanTiles tiles: the tile counts (of count_kernel, or counted here for at
// most kScanCountTiles tiles) -> tile offsets, and the per-request metadata.  Invalid cu_seqlens: reported, num_actual_tokens = 0 and no per-request
// metadata; the tile offsets depend only on the mask and T, so they are still written and the gather
// launched after this kernel stays in bounds whatever cu_seqlens holds.
__global__ void __launch_bounds__(1024) scan_kernel(const uint8_t* __restrict__ keep, const int32_t* __restrict__ cu,
                                                    int R, int T, int* tile_cnt, int* tile_off,
                                                    int32_t* new_cu, int32_t* new_len, int32_t* num_actual,
                                                    int32_t* kept_len, uint8_t* drop_layer, int L, int layer,
                                                    int32_t* status, int count_here) {
    pdl_wait();
    pdl_trigger();
    __shared__ int sh[32];
    __shared__ int s_bad;
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const bool ok = cu_valid(cu, R, T, &s_bad);
    if (!ok && tid == 0) {
        set_status(status, UP_DEV_BAD_CU_SEQLENS);
        *num_actual = 0;
    }
    const int tiles = (T + kTile - 1) / kTile;
    if (count_here) {
        // a short stream (tiles <= kScanCountTiles): one warp per tile, 16 flags per lane and load
        for (int i = w; i < tiles; i += blockDim.x / 32) {
            int c = 0;
            for (int j = lane; j < kTile / 16; j += 32) {
                const int64_t t = (int64_t)i * kTile + j * 16;
                if (t < T) c += count_nonzero_bytes(load_flags16(keep, t, T));
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
            if (lane == 0 && UP_IN(i, tiles, status)) tile_cnt[i] = c;
        }
        __syncthreads();
    }
    // exclusive scan of the tile counts (tiles split in contiguous chunks over the threads)
    const int per = (tiles + blockDim.x - 1) / blockDim.x;
    const int a0 = min(tiles, tid * per), a1 = min(tiles, a0 + per);
    int local = 0;
    for (int i = a0; i < a1; ++i) local += UP_IN(i, tiles, status) ? tile_cnt[i] : 0;
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
    const int total = sh[31];
    int off = (w > 0 ? sh[w - 1] : 0) + x - local;
    for (int i = a0; i < a1; ++i) {
        if (!UP_IN(i, tiles, status)) continue;
        tile_off[i] = off;
        off += tile_cnt[i];
    }
    __syncthreads();
    if (!ok) return;
    request_metadata(keep, cu, R, T, tiles, tile_off, total, new_cu, new_len, num_actual, kept_len, drop_layer, L, layer,
                     status);
}

// One warp copies one row of V 16-byte vectors, kRowUnroll loads in flight per lane.  In the
// bounds-checked build the callers check the two row indices first.
__device__ __forceinline__ void copy_row(const uint4* __restrict__ s, uint4* __restrict__ d, int V, int lane) {
    int j = lane;
    for (; j + 32 * (kRowUnroll - 1) < V; j += 32 * kRowUnroll) {
        uint4 r[kRowUnroll];
#pragma unroll
        for (int u = 0; u < kRowUnroll; ++u) r[u] = __ldcs(s + j + 32 * u);
#pragma unroll
        for (int u = 0; u < kRowUnroll; ++u) d[j + 32 * u] = r[u];
    }
    for (; j < V; j += 32) d[j] = __ldcs(s + j);
}

// Items (tile, part) = (item / parts, item % parts), visited round-robin by the persistent CTAs: the
// tile's kept tokens in ascending order (a scan of its 1024 flags, recomputed by every part), the
// index/positions/slots rows written by part 0, and the part's contiguous share of the kept hidden rows
// copied.
// Metadata outputs of a gather that scans the stream itself (SELF).
struct MetaOut {
    const int32_t* cu;
    int R, L, layer;
    int32_t *new_cu, *new_len, *num_actual, *kept_len, *status;
    uint8_t* drop_layer;
};

// SELF (streams of at most kSelfScanTiles tiles, one launch for the whole compaction): every CTA
// counts the tiles (one warp per tile) and scans the counts into shared memory instead of reading the
// scan kernel's tile_off, and CTA 0 also validates cu_seqlens and writes the per-request metadata.
template <bool ROWS, bool SELF>
__global__ void __launch_bounds__(kGatherThreads) gather_kernel(const uint8_t* __restrict__ keep, int T, int tiles,
                                                              int parts, const int* __restrict__ tile_off,
                                                              const int64_t* __restrict__ pos,
                                                              const int64_t* __restrict__ slots, int32_t* kept_index,
                                                              int64_t* out_pos, int64_t* out_slots,
                                                              const uint4* __restrict__ src, uint4* __restrict__ dst,
                                                              int V, MetaOut M) {
    pdl_wait();
    pdl_trigger();
    __shared__ int s_src[kTile];           // source token of the tile's k-th kept token
    __shared__ int s_wsum[kTileThreads / 32];
    __shared__ int s_off[kSelfScanTiles];
    __shared__ int s_total, s_bad;
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    if (SELF) {
        for (int i = w; i < tiles; i += kGatherThreads / 32) {
            int c = 0;
            for (int j = lane; j < kTile / 16; j += 32) {
                const int64_t t = (int64_t)i * kTile + j * 16;
                if (t < T) c += count_nonzero_bytes(load_flags16(keep, t, T));
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
            if (lane == 0) s_off[i] = c;
        }
        __syncthreads();
        if (w == 0) {                      // exclusive scan of <= 8 counts
            const int x0 = 2 * lane < tiles ? s_off[2 * lane] : 0;
            const int x1 = 2 * lane + 1 < tiles ? s_off[2 * lane + 1] : 0;
            int x = x0 + x1;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, x, o);
                if (lane >= o) x += y;
            }
            const int e = x - x0 - x1;
            __syncwarp();
            if (2 * lane < tiles) s_off[2 * lane] = e;
            if (2 * lane + 1 < tiles) s_off[2 * lane + 1] = e + x0;
            if (lane == 31) s_total = x;
        }
        __syncthreads();
        if (blockIdx.x == 0) {
            if (cu_valid(M.cu, M.R, T, &s_bad))
                request_metadata(keep, M.cu, M.R, T, tiles, s_off, s_total, M.new_cu, M.new_len, M.num_actual,
                                 M.kept_len, M.drop_layer, M.L, M.layer, M.status);
            else if (tid == 0) {
                set_status(M.status, UP_DEV_BAD_CU_SEQLENS);
                *M.num_actual = 0;
            }
        }
    }
    const int64_t items = (int64_t)tiles * parts;
    for (int64_t item = blockIdx.x; item < items; item += gridDim.x) {
        const int tile = static_cast<int>(item / parts), part = static_cast<int>(item % parts);
        const int64_t t0 = (int64_t)tile * kTile + tid * 16;         // threads 0..63 own 16 flags each
        uint4 f = make_uint4(0, 0, 0, 0);
        if (tid < kTileThreads && t0 < T) f = load_flags16(keep, t0, T);
        const int c = count_nonzero_bytes(f);
        int x = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        __syncthreads();                    // the previous item is done with s_src and s_wsum
        if (lane == 31 && w < kTileThreads / 32) s_wsum[w] = x;
        __syncthreads();
        if (tid < kTileThreads) {
            int d = x - c;
            for (int i = 0; i < w; ++i) d += s_wsum[i];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const uint32_t wv = i < 4 ? f.x : i < 8 ? f.y : i < 12 ? f.z : f.w;
                if ((wv >> (8 * (i & 3))) & 0xFFu) s_src[d++] = static_cast<int>(t0 + i);
            }
        }
        int cnt = 0;
#pragma unroll
        for (int i = 0; i < kTileThreads / 32; ++i) cnt += s_wsum[i];
        __syncthreads();
        const int base = SELF ? s_off[tile] : (UP_IN(tile, tiles, M.status) ? tile_off[tile] : 0);
        if (part == 0) {
            for (int k = tid; k < cnt; k += kGatherThreads) {
                const int sidx = s_src[k];
                if (!UP_IN(base + k, T, M.status) || !UP_IN(sidx, T, M.status)) continue;
                kept_index[base + k] = sidx;
                if (out_pos) out_pos[base + k] = pos[sidx];
                if (out_slots) out_slots[base + k] = slots[sidx];
            }
        }
        if (ROWS) {
            const int per = (cnt + parts - 1) / parts;
            const int k0 = part * per, k1 = min(cnt, k0 + per);
            for (int k = k0 + w; k < k1; k += kGatherThreads / 32)
                if (UP_IN(s_src[k], T, M.status) && UP_IN(base + k, T, M.status))
                    copy_row(src + (int64_t)s_src[k] * V, dst + (int64_t)(base + k) * V, V, lane);
        }
    }
}

// dst[row_d(k)] = src[row_s(k)] for k < *count; one warp per row, 16-byte vectors
template <bool GATHER>
__global__ void __launch_bounds__(kRowThreads) rows_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                                           const int32_t* __restrict__ idx,
                                                           const int32_t* __restrict__ count, int64_t T_upper,
                                                           int V, int32_t* status) {
    pdl_wait();
    pdl_trigger();
    const int n = *count;
    if (n < 0 || n > T_upper) {
        if (blockIdx.x == 0 && threadIdx.x == 0) set_status(status, UP_DEV_BAD_TOKEN_COUNT);
        return;
    }
    const int lane = threadIdx.x & 31;
    const int warps = gridDim.x * (kRowThreads / 32);
    for (int k = blockIdx.x * (kRowThreads / 32) + (threadIdx.x >> 5); k < n; k += warps) {
        const int64_t other = idx[k];
        // the residual's row count is not an argument: the bounds-checked build checks the sign only
        if (!UP_IN(other, int64_t(1) << 31, status)) continue;
        copy_row(src + (GATHER ? other : (int64_t)k) * V, dst + (GATHER ? (int64_t)k : other) * V, V, lane);
    }
}

// CTAs of a kernel that are resident on the whole GPU at once (occupancy x SMs), once per process: a
// persistent grid of exactly this size runs in one wave.
template <typename K>
static int resident_ctas(K kernel, int threads) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, 0) != cudaSuccess || per_sm <= 0)
        per_sm = 1;
    return per_sm * num_sms();
}
static int scatter_resident() {
    static int n = 0;
    static std::once_flag once;
    std::call_once(once, [] { n = resident_ctas(rows_kernel<false>, kRowThreads); });
    return n;
}

// CTAs of gather_kernel that are resident on the whole GPU at once (occupancy x SMs), once per process.
template <bool ROWS, bool SELF>
static int gather_resident() {
    static int n = 0;
    static std::once_flag once;
    std::call_once(once, [] { n = resident_ctas(gather_kernel<ROWS, SELF>, kGatherThreads); });
    return n;
}

template <bool SELF>
static void launch_gather(const uint8_t* keep, int Ti, int tiles, const int* tile_off, const uint16_t* hidden,
                          int hdim, const int64_t* positions, const int64_t* slots, uint16_t* out_hidden,
                          int64_t* out_positions, int64_t* out_slots, int32_t* kept_index, const MetaOut& M,
                          cudaStream_t st) {
    // persistent CTAs: as many as fit on the GPU at once; parts per tile so that every resident CTA
    // has about kItemsPerCta items, which keeps the last round (the CTAs that get one item more than
    // the others) to a few percent of the copy (4 items per CTA measured 2% slower on 64 x 32K tokens)
    const int resident = hidden ? gather_resident<true, SELF>() : gather_resident<false, SELF>();
    const int parts = hidden ? static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(kMaxParts, cdiv((int64_t)kItemsPerCta * resident, std::max(1, tiles)))))
                             : 1;
    const int grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>((int64_t)tiles * parts, resident)));
    if (hidden)
        launch_pdl(gather_kernel<true, SELF>, dim3(grid), dim3(kGatherThreads), 0, st,
            keep, Ti, tiles, parts, tile_off, positions, slots, kept_index, out_positions, out_slots,
            reinterpret_cast<const uint4*>(hidden), reinterpret_cast<uint4*>(out_hidden), hdim / 8, M);
    else
        launch_pdl(gather_kernel<false, SELF>, dim3(grid), dim3(kGatherThreads), 0, st,
            keep, Ti, tiles, 1, tile_off, positions, slots, kept_index, out_positions, out_slots, nullptr,
            nullptr, 0, M);
    count_launch();
}

// The launches of one compaction, on the caller's workspace or the fixed scratch alike.
static void launch_compaction(const uint8_t* keep, const int32_t* cu, int R, int Ti, const uint16_t* hidden,
                              int hdim, const int64_t* positions, const int64_t* slots, uint16_t* out_hidden,
                              int64_t* out_positions, int64_t* out_slots, int32_t* kept_index, int32_t* new_cu,
                              int32_t* new_len, int32_t* num_actual, int32_t* kept_len, uint8_t* drop_layer,
                              int L, int layer, int* tile_cnt, int* tile_off, int32_t* status, cudaStream_t st) {
    const int tiles = static_cast<int>(cdiv(Ti, kTile));
    const MetaOut M{cu, R, L, layer, new_cu, new_len, num_actual, kept_len, status, drop_layer};
    if (tiles <= kSelfScanTiles) {        // one launch: the gather scans the short stream itself
        launch_gather<true>(keep, Ti, tiles, nullptr, hidden, hdim, positions, slots, out_hidden, out_positions,
                            out_slots, kept_index, M, st);
        return;
    }
    const int count_here = tiles <= kScanCountTiles ? 1 : 0;
    if (!count_here) {
        launch_pdl(count_kernel, dim3(tiles), dim3(kTileThreads), 0, st, keep, Ti, tile_cnt, tiles, status);
        count_launch();
    }
    launch_pdl(scan_kernel, dim3(1), dim3(1024), 0, st,
        keep, cu, R, Ti, tile_cnt, tile_off, new_cu, new_len, num_actual, kept_len, drop_layer, L, layer, status,
        count_here);
    count_launch();
    launch_gather<false>(keep, Ti, tiles, tile_off, hidden, hdim, positions, slots, out_hidden, out_positions,
                         out_slots, kept_index, M, st);
}

}  // namespace compact
}  // namespace up

using namespace up;

extern "C" size_t up_compact_workspace_bytes(int R, int64_t T) {
    if (R <= 0 || T < 0 || T >= (int64_t(1) << 31)) return 0;
    return compact::layout(T).total;
}

extern "C" up_status up_compact(const uint8_t* token_keep, const int32_t* cu_seqlens, int R, int64_t T,
                                const uint16_t* hidden, int hdim, const int64_t* positions, const int64_t* slots,
                                uint16_t* out_hidden, int64_t* out_positions, int64_t* out_slots,
                                int32_t* kept_index, int32_t* new_cu_seqlens, int32_t* new_seq_lens,
                                int32_t* num_actual_tokens, int32_t* kept_len, uint8_t* drop_layer, int L, int layer,
                                void* ws, size_t ws_bytes, int32_t* dev_status, void* stream) {
    // token_keep may be NULL for a batch without tokens (T = 0)
    if ((T > 0 && !token_keep) || !cu_seqlens || !kept_index || !new_cu_seqlens || !new_seq_lens ||
        !num_actual_tokens || !ws || !dev_status)
        return UP_ERR_ARG;
    if (R <= 0 || T < 0 || T >= (int64_t(1) << 31)) return UP_ERR_ARG;
    if ((hidden == nullptr) != (out_hidden == nullptr) || (positions == nullptr) != (out_positions == nullptr) ||
        (slots == nullptr) != (out_slots == nullptr))
        return UP_ERR_ARG;
    if ((kept_len || drop_layer) && (layer < 0 || layer >= L)) return UP_ERR_ARG;
    if (hidden && (hdim <= 0 || hdim % 8 != 0 || !aligned16(hidden) || !aligned16(out_hidden))) return UP_ERR_SHAPE;
    if (!aligned16(token_keep) || !aligned16(ws)) return UP_ERR_SHAPE;
    const compact::Layout Lw = compact::layout(T);
    if (ws_bytes < Lw.total) return UP_ERR_WORKSPACE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int* tile_cnt = reinterpret_cast<int*>(static_cast<uint8_t*>(ws) + Lw.tile_cnt);
    int* tile_off = reinterpret_cast<int*>(static_cast<uint8_t*>(ws) + Lw.tile_off);
    compact::launch_compaction(token_keep, cu_seqlens, R, static_cast<int>(T), hidden, hdim, positions, slots,
                               out_hidden, out_positions, out_slots, kept_index, new_cu_seqlens, new_seq_lens,
                               num_actual_tokens, kept_len, drop_layer, L, layer, tile_cnt, tile_off, dev_status, st);
    return check_launch();
}

extern "C" up_status up_scatter_back(const uint16_t* new_states, const int32_t* kept_index,
                                     const int32_t* num_actual_tokens, int64_t T_upper, int hdim, uint16_t* residual,
                                     int32_t* dev_status, void* stream) {
    if (T_upper < 0 || T_upper >= (int64_t(1) << 31)) return UP_ERR_ARG;
    if (hdim <= 0 || hdim % 8 != 0) return UP_ERR_SHAPE;
    if (T_upper == 0) return UP_OK;        // no rows: the buffers may be empty (NULL)
    if (!new_states || !kept_index || !num_actual_tokens || !residual || !dev_status) return UP_ERR_ARG;
    if (!aligned16(new_states) || !aligned16(residual)) return UP_ERR_SHAPE;
    const int V = hdim / 8;
    // one wave of persistent CTAs (a grid larger than what is resident leaves a trailing partial wave)
    const int grid = static_cast<int>(
        std::max<int64_t>(1, std::min<int64_t>(cdiv(T_upper, compact::kRowThreads / 32), compact::scatter_resident())));
    launch_pdl(compact::rows_kernel<false>, dim3(grid), dim3(compact::kRowThreads), 0, static_cast<cudaStream_t>(stream),
        reinterpret_cast<const uint4*>(new_states), reinterpret_cast<uint4*>(residual), kept_index,
        num_actual_tokens, T_upper, V, dev_status);
    count_launch();
    return check_launch();
}

// ------------------------------------------------------------------------------------------------
// Compaction without a caller workspace.
//
// Some callers cannot hand this library a scratch buffer: an inference engine whose memory planner
// owns every byte of device memory after start-up, a plugin host that only passes in the tensors it
// already has, or a latency-critical loop that must never hit cudaMalloc's implicit device
// synchronisation.  For them up_compact_noalloc keeps the per-tile counts and offsets in a
// fixed-size array that is part of this library's device image: it exists on every GPU that loads
// the library, from load time until the process exits, and nothing is allocated per call.

namespace up {
namespace compact {

constexpr int kNoAllocMaxTiles = UP_NOALLOC_MAX_TOKENS / kTile;        // 16384 tiles of 1024 tokens
static_assert(UP_NOALLOC_MAX_TOKENS % kTile == 0, "the token limit must be whole tiles");

// [0, kNoAllocMaxTiles + 1): tile counts; [kNoAllocMaxTiles + 1, 2 * (kNoAllocMaxTiles + 1)): offsets.
// Every call overwrites every entry it reads, so nothing here needs clearing between calls.
static __device__ __align__(256) int g_noalloc_scratch[2 * (kNoAllocMaxTiles + 1)];

// Device address of g_noalloc_scratch on the current device (the host-side symbol is only a handle),
// looked up once per device with that device current.
static int* noalloc_scratch(up_status* err) {
    static int* addr[64] = {nullptr};
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        *err = UP_ERR_CUDA;
        return nullptr;
    }
    std::lock_guard<std::mutex> lk(mu);
    if (addr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
            *err = UP_ERR_CUDA;
            return nullptr;
        }
        addr[dev] = static_cast<int*>(p);
    }
    *err = UP_OK;
    return addr[dev];
}

}  // namespace compact
}  // namespace up

extern "C" up_status up_compact_noalloc(const uint8_t* token_keep, const int32_t* cu_seqlens, int R, int64_t T,
                                        const uint16_t* hidden, int hdim, const int64_t* positions,
                                        const int64_t* slots, uint16_t* out_hidden, int64_t* out_positions,
                                        int64_t* out_slots, int32_t* kept_index, int32_t* new_cu_seqlens,
                                        int32_t* new_seq_lens, int32_t* num_actual_tokens, int32_t* kept_len,
                                        uint8_t* drop_layer, int L, int layer, int32_t* dev_status, void* stream) {
    if ((T > 0 && !token_keep) || !cu_seqlens || !kept_index || !new_cu_seqlens || !new_seq_lens ||
        !num_actual_tokens || !dev_status)
        return UP_ERR_ARG;
    if (R <= 0 || T < 0 || T >= (int64_t(1) << 31)) return UP_ERR_ARG;
    if (T > UP_NOALLOC_MAX_TOKENS) return UP_ERR_WORKSPACE;     // beyond the fixed scratch: use up_compact
    if ((hidden == nullptr) != (out_hidden == nullptr) || (positions == nullptr) != (out_positions == nullptr) ||
        (slots == nullptr) != (out_slots == nullptr))
        return UP_ERR_ARG;
    if ((kept_len || drop_layer) && (layer < 0 || layer >= L)) return UP_ERR_ARG;
    if (hidden && (hdim <= 0 || hdim % 8 != 0 || !aligned16(hidden) || !aligned16(out_hidden))) return UP_ERR_SHAPE;
    if (!aligned16(token_keep)) return UP_ERR_SHAPE;
    up_status err;
    int* scratch = compact::noalloc_scratch(&err);
    if (scratch == nullptr) return err;
    int* tile_cnt = scratch;
    int* tile_off = scratch + compact::kNoAllocMaxTiles + 1;
    compact::launch_compaction(token_keep, cu_seqlens, R, static_cast<int>(T), hidden, hdim, positions, slots,
                               out_hidden, out_positions, out_slots, kept_index, new_cu_seqlens, new_seq_lens,
                               num_actual_tokens, kept_len, drop_layer, L, layer, tile_cnt, tile_off, dev_status,
                               static_cast<cudaStream_t>(stream));
    return check_launch();
}
