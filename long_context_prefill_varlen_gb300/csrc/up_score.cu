// up_score_blocks: block-level importance of UniPrefill ("UniPrefill: Universal Long-Context
// Prefill Acceleration via Block-wise Dynamic Sparsification", arXiv 2605.06221, section 3.2,
// Eqs. 2-4, and the kernel pipeline of section 3.5, Eq. 13).
//
// For every request r, KV head kh and the group x n window query rows that read kh:
//   pass 1  S = Qwin . K^T on tcgen05 (query rows in TMEM lanes, 128 keys per tile in columns);
//           per row the online max m and sum l of 2^(S*a - m) over the causal key range;
//           per work item (kItemTiles key tiles) a partial (m, l); the last CTA of each
//           (r, kh, slab) unit merges the partials in a fixed order into c = m + log2(l).
//   pass 2  S^T = K . Qwin^T (128 keys in TMEM lanes, query rows in columns); each thread owns a
//           key and sums P = 2^(S*a - c_row) over its rows; the per-key sums are reduced over G
//           consecutive keys with warp shuffles and written as per-(unit, block) partials.
//   final   b_g = (sum over units of the partials) / (n_eff * Hq * G).
// a = sm_scale * log2(e): the softmax is computed in base 2, exactly equal to exp in base e.
//
// CTA layout (320 threads, one CTA per SM, persistent over a contiguous range of work items):
//   warp 0   TMA producer: the query slab of the current unit, then K tiles into a 5-stage ring
//   warp 1   TMEM allocator and single-thread tcgen05.mma issuer
//   warps 2-9  two epilogue warpgroups; warpgroup w reads TMEM columns [64w, 64w+64) of every
//              128x128 accumulator, so both share each job (a job = one 128x128 MMA tile)
// TMEM: 4 accumulators of 128 columns (the whole 512-column TMEM), used as a ring of jobs.
#include <math.h>

#include <algorithm>
#include <mutex>

#include "up_internal.cuh"

namespace up {
namespace score {

constexpr int kTileKeys = 128;
constexpr int kStageBytes = 128 * 128;          // 128 rows x 64 bf16 (one 128-byte swizzle atom wide)
constexpr int kStages = 5;
constexpr int kSlabBytes = 128 * 1024;          // resident query rows of one unit
constexpr int kItemTiles = 2;                   // key tiles per work item (pass-1 partial granularity)
constexpr int kThreads = 320;
constexpr int kMaxJ = 8;                        // 128-row jobs per slab (d_k = 64 -> 8)
constexpr int kTmemCols = 512;
constexpr uint32_t kIdesc = idesc_bf16_f32(128, 128);
constexpr int kCtrlBytes = 256;
constexpr int kCvecFloats = 1024;
constexpr int kXchgBytes = kMaxJ * 128 * 8;
constexpr int kSmemBytes = 1024 + kSlabBytes + kStages * kStageBytes + kCtrlBytes + kCvecFloats * 4 + kXchgBytes;

struct Geometry {
    int group, rows_total, slab_rows, slabs, J, box_rows, nc;
};

struct Layout {
    size_t items, unit_items, n_items, unit_done, ml, cvec, blk, tok, total;
    int64_t items_cap, units;
};

struct Params {
    const int32_t* cu;
    const int32_t* cb;
    int R, T, Hq, Hkv, dk, G, n, group, rows_total, slab_rows, slabs, J, box_rows, units_per_req;
    float a;
    int64_t nb_cap;
    int4* items;
    int2* unit_items;
    int* n_items;
    int* unit_done;
    float2* ml;
    float* cvec;
    float* blk;
    float* tok;
    float* block_scores;
    float* token_scores;
    int32_t* status;
};

static bool geometry(int Hq, int Hkv, int dk, int n, Geometry* g) {
    if (Hq <= 0 || Hkv <= 0 || Hq % Hkv) return false;
    if (dk != 64 && dk != 128 && dk != 256) return false;
    const bool small_n = (n == 16 || n == 32 || n == 64 || n == 128);
    const bool big_n = (n > 128 && n <= 1024 && n % 128 == 0);
    if (!small_n && !big_n) return false;
    g->group = Hq / Hkv;
    g->rows_total = g->group * n;
    const int max_rows = kSlabBytes / (dk * 2);
    g->slab_rows = std::min<int>(static_cast<int>(cdiv(g->rows_total, 128) * 128), max_rows);
    g->slabs = static_cast<int>(cdiv(g->rows_total, g->slab_rows));
    g->J = g->slab_rows / 128;
    g->box_rows = std::min(n, 128);
    g->nc = dk / 64;
    return g->J <= kMaxJ && (g->nc < 4 || g->J <= 2);
}

static Layout layout(int R, int64_t T, const Geometry& g, int Hkv, int64_t nb_cap, bool tok) {
    Layout L{};
    L.items_cap = (cdiv(T, (int64_t)kTileKeys * kItemTiles) + R) * Hkv * g.slabs;
    L.units = (int64_t)R * Hkv * g.slabs;
    size_t o = 0;
    auto take = [&](size_t bytes) { size_t at = o; o = align_up(o + bytes, 256); return at; };
    L.items = take(sizeof(int4) * L.items_cap);
    L.unit_items = take(sizeof(int2) * L.units);
    L.n_items = take(16);
    L.unit_done = take(sizeof(int) * L.units);
    L.ml = take(sizeof(float2) * L.items_cap * g.slab_rows);
    L.cvec = take(sizeof(float) * L.units * g.slab_rows);
    L.blk = take(sizeof(float) * (size_t)Hkv * g.slabs * nb_cap);
    L.tok = tok ? take(sizeof(float) * (size_t)Hkv * g.slabs * T) : 0;
    L.total = o;
    return L;
}

// ------------------------------------------------------------------------------------------------
// plan: validate the varlen metadata and lay out the work items (one CTA)

__device__ __forceinline__ int block_exclusive_scan_1024(int v, int* sh, int* total) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) sh[w] = x;
    __syncthreads();
    if (w == 0) {
        int s = sh[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o) s += y;
        }
        sh[lane] = s;   // inclusive over warps
    }
    __syncthreads();
    const int before = (w > 0 ? sh[w - 1] : 0) + x - v;
    *total = sh[31];
    __syncthreads();
    return before;
}

__global__ void __launch_bounds__(1024) plan_kernel(Params P) {
    __shared__ int s_bad;
    __shared__ int s_scan[32];
    const int tid = threadIdx.x;
    if (tid == 0) s_bad = 0;
    __syncthreads();
    for (int r = tid; r < P.R; r += blockDim.x) {
        const int c0 = P.cu[r], c1 = P.cu[r + 1];
        if ((r == 0 && c0 != 0) || c1 < c0 || c1 > P.T || (r == P.R - 1 && c1 != P.T)) atomicOr(&s_bad, 1);
        const int nb = (c1 - c0 + P.G - 1) / P.G;
        const int b0 = P.cb[r], b1 = P.cb[r + 1];
        if ((r == 0 && b0 != 0) || b1 - b0 != nb || (int64_t)b1 > P.nb_cap) atomicOr(&s_bad, 2);
    }
    __syncthreads();
    if (s_bad) {
        if (tid == 0) {
            set_status(P.status, (s_bad & 1) ? UP_DEV_BAD_CU_SEQLENS : UP_DEV_BAD_CU_BLOCKS);
            P.n_items[0] = 0;
            P.n_items[1] = 0;      // metadata invalid: finalize writes nothing
        }
        return;
    }
    const int per = (P.R + blockDim.x - 1) / blockDim.x;
    const int r0 = min(P.R, tid * per), r1 = min(P.R, r0 + per);
    auto nitems = [&](int r) {
        const int N = P.cu[r + 1] - P.cu[r];
        const int ntiles = (N + kTileKeys - 1) / kTileKeys;
        return (ntiles + kItemTiles - 1) / kItemTiles;
    };
    int local = 0;
    for (int r = r0; r < r1; ++r) local += nitems(r) * P.units_per_req;
    int total = 0;
    int off = block_exclusive_scan_1024(local, s_scan, &total);
    for (int r = r0; r < r1; ++r) {
        const int N = P.cu[r + 1] - P.cu[r];
        const int ntiles = (N + kTileKeys - 1) / kTileKeys;
        const int ni = nitems(r);
        for (int kk = 0; kk < P.units_per_req; ++kk) {
            const int u = r * P.units_per_req + kk;
            P.unit_items[u] = make_int2(off + kk * ni, ni);
            P.unit_done[u] = 0;
            for (int s = 0; s < ni; ++s)
                P.items[off + kk * ni + s] = make_int4(r, kk, s * kItemTiles, min(ntiles, (s + 1) * kItemTiles));
        }
        off += ni * P.units_per_req;
    }
    if (tid == 0) {
        P.n_items[0] = total;
        P.n_items[1] = 1;          // metadata validated
    }
}

// ------------------------------------------------------------------------------------------------
// the two tcgen05 passes

struct Smem {
    uint8_t* slab;
    uint8_t* stages;
    uint64_t* full;        // [kStages]  TMA landed
    uint64_t* empty;       // [kStages]  MMAs done reading the stage
    uint64_t* tfull;       // [4]        accumulator ready
    uint64_t* tempty;      // [4]        accumulator drained by both warpgroups
    uint64_t* slab_full;
    uint64_t* slab_free;
    uint64_t* mma_done;
    uint32_t* tmem_holder;
    int* abort_flag;
    int* last_flag;
    float* cvec;           // [kCvecFloats]
    uint8_t* xchg;         // [kXchgBytes]
};

__device__ __forceinline__ Smem carve(uint8_t* raw) {
    Smem s;
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    s.slab = base;
    s.stages = base + kSlabBytes;
    uint8_t* ctrl = s.stages + kStages * kStageBytes;
    uint64_t* b = reinterpret_cast<uint64_t*>(ctrl);
    s.full = b;
    s.empty = b + kStages;
    s.tfull = b + 2 * kStages;
    s.tempty = b + 2 * kStages + 4;
    s.slab_full = b + 2 * kStages + 8;
    s.slab_free = b + 2 * kStages + 9;
    s.mma_done = b + 2 * kStages + 10;
    s.tmem_holder = reinterpret_cast<uint32_t*>(b + 2 * kStages + 11);
    s.abort_flag = reinterpret_cast<int*>(s.tmem_holder + 1);
    s.last_flag = s.abort_flag + 1;
    s.cvec = reinterpret_cast<float*>(ctrl + kCtrlBytes);
    s.xchg = reinterpret_cast<uint8_t*>(s.cvec + kCvecFloats);
    return s;
}

struct ItemInfo {
    int r, kk, tb, te, unit, base, N, kh, slab;
};

__device__ __forceinline__ ItemInfo item_info(const Params& P, int it) {
    const int4 w = P.items[it];
    ItemInfo I;
    I.r = w.x;
    I.kk = w.y;
    I.tb = w.z;
    I.te = w.w;
    I.unit = I.r * P.units_per_req + I.kk;
    I.base = P.cu[I.r];
    I.N = P.cu[I.r + 1] - I.base;
    I.kh = I.kk / P.slabs;
    I.slab = I.kk % P.slabs;
    return I;
}

// Bounded drain used only after an abort: wait for the loads this thread issued to land, so no
// TMA write can reach shared memory after the CTA exits.
__device__ void drain_loads(const Smem& S, uint32_t stage_cnt, uint32_t slab_cnt) {
    const uint64_t t0 = globaltimer_ns();
    const uint32_t first = stage_cnt > kStages ? stage_cnt - kStages : 0;
    for (uint32_t sc = first; sc < stage_cnt; ++sc)
        while (!mbar_try_wait(smem_u32(S.full + sc % kStages), (sc / kStages) & 1))
            if (globaltimer_ns() - t0 > kWaitLimitNs) return;
    if (slab_cnt > 0)
        while (!mbar_try_wait(smem_u32(S.slab_full), (slab_cnt - 1) & 1))
            if (globaltimer_ns() - t0 > kWaitLimitNs) return;
}

template <int NC>
__device__ void producer(const Params& P, const Smem& S, const CUtensorMap* tmQ, const CUtensorMap* tmK,
                         int it0, int it1) {
    volatile int* abort_flag = S.abort_flag;
    int prev_unit = -1;
    uint32_t stage_cnt = 0, slab_cnt = 0;
    const uint32_t slab_addr = smem_u32(S.slab), stage_addr = smem_u32(S.stages);
    for (int it = it0; it < it1; ++it) {
        const ItemInfo I = item_info(P, it);
        if (I.unit != prev_unit) {
            if (!mbar_wait(smem_u32(S.slab_free), (slab_cnt & 1) ^ 1, abort_flag)) {
                drain_loads(S, stage_cnt, slab_cnt);
                return;
            }
            const int row0 = I.slab * P.slab_rows;
            const int rows = min(P.slab_rows, P.rows_total - row0);
            const uint32_t bar = smem_u32(S.slab_full);
            mbar_arrive_expect_tx(bar, static_cast<uint32_t>(rows) * NC * 128u);
            for (int qr = 0; qr < rows; qr += P.box_rows) {
                const int qg = row0 + qr;
                const int hl = qg / P.n, t0 = qg % P.n;
                const int head = I.kh * P.group + hl;
                const int tok = I.base + I.N - P.n + t0;      // may be < 0: TMA fills zeros
#pragma unroll
                for (int c = 0; c < NC; ++c)
                    tma_load_3d(slab_addr + c * P.slab_rows * 128 + qr * 128, tmQ, bar, c * 64, head, tok);
            }
            ++slab_cnt;
            prev_unit = I.unit;
        }
        for (int kt = I.tb; kt < I.te; ++kt) {
#pragma unroll
            for (int c = 0; c < NC; ++c) {
                const uint32_t s = stage_cnt % kStages, ph = (stage_cnt / kStages) & 1;
                if (!mbar_wait(smem_u32(S.empty + s), ph ^ 1, abort_flag)) {
                    drain_loads(S, stage_cnt, slab_cnt);
                    return;
                }
                mbar_arrive_expect_tx(smem_u32(S.full + s), kStageBytes);
                tma_load_3d(stage_addr + s * kStageBytes, tmK, smem_u32(S.full + s), c * 64, I.kh,
                            I.base + kt * kTileKeys);
                ++stage_cnt;
            }
        }
    }
}

template <int PASS, int NC>
__device__ void mma_issuer(const Params& P, const Smem& S, uint32_t tmem_base, int it0, int it1) {
    volatile int* abort_flag = S.abort_flag;
    int prev_unit = -1;
    uint32_t stage_cnt = 0, slab_cnt = 0, jc = 0;
    const uint32_t slab_addr = smem_u32(S.slab), stage_addr = smem_u32(S.stages);
    const int J = P.J;
    auto slab_desc = [&](int j, int c, int k) {   // 128 query rows of job j, k-chunk c, 16-wide slice k
        return sdesc_sw128(slab_addr + c * P.slab_rows * 128 + j * 128 * 128 + k * 32);
    };
    auto stage_desc = [&](uint32_t s, int k) { return sdesc_sw128(stage_addr + s * kStageBytes + k * 32); };
    for (int it = it0; it < it1; ++it) {
        const ItemInfo I = item_info(P, it);
        if (I.unit != prev_unit) {
            if (prev_unit >= 0) tc_commit(smem_u32(S.slab_free));
            if (!mbar_wait(smem_u32(S.slab_full), slab_cnt & 1, abort_flag)) goto out;
            ++slab_cnt;
            tc_fence_after();
            prev_unit = I.unit;
        }
        for (int kt = I.tb; kt < I.te; ++kt) {
            if (NC <= 2) {
                // jobs outer: the tile's K stages stay resident while the J jobs run
                for (int j = 0; j < J; ++j) {
                    const uint32_t buf = jc & 3;
                    if (!mbar_wait(smem_u32(S.tempty + buf), ((jc >> 2) & 1) ^ 1, abort_flag)) goto out;
                    tc_fence_after();
#pragma unroll
                    for (int c = 0; c < NC; ++c) {
                        const uint32_t sc = stage_cnt + c, s = sc % kStages;
                        if (j == 0) {
                            if (!mbar_wait(smem_u32(S.full + s), (sc / kStages) & 1, abort_flag)) goto out;
                            tc_fence_after();
                        }
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const uint64_t a = PASS == 1 ? slab_desc(j, c, k) : stage_desc(s, k);
                            const uint64_t b = PASS == 1 ? stage_desc(s, k) : slab_desc(j, c, k);
                            tc_mma_bf16(tmem_base + buf * 128, a, b, kIdesc, (c | k) != 0);
                        }
                    }
                    tc_commit(smem_u32(S.tfull + buf));
                    ++jc;
                }
#pragma unroll
                for (int c = 0; c < NC; ++c) tc_commit(smem_u32(S.empty + (stage_cnt + c) % kStages));
                stage_cnt += NC;
            } else {
                // chunks outer (d_k = 256, J <= 2): each K stage is released as soon as all jobs used it
                for (int j = 0; j < J; ++j) {
                    const uint32_t q = jc + j;
                    if (!mbar_wait(smem_u32(S.tempty + (q & 3)), ((q >> 2) & 1) ^ 1, abort_flag)) goto out;
                }
                tc_fence_after();
#pragma unroll
                for (int c = 0; c < NC; ++c) {
                    const uint32_t s = stage_cnt % kStages;
                    if (!mbar_wait(smem_u32(S.full + s), (stage_cnt / kStages) & 1, abort_flag)) goto out;
                    tc_fence_after();
                    for (int j = 0; j < J; ++j) {
                        const uint32_t buf = (jc + j) & 3;
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const uint64_t a = PASS == 1 ? slab_desc(j, c, k) : stage_desc(s, k);
                            const uint64_t b = PASS == 1 ? stage_desc(s, k) : slab_desc(j, c, k);
                            tc_mma_bf16(tmem_base + buf * 128, a, b, kIdesc, (c | k) != 0);
                        }
                    }
                    tc_commit(smem_u32(S.empty + s));
                    ++stage_cnt;
                }
                for (int j = 0; j < J; ++j) tc_commit(smem_u32(S.tfull + ((jc + j) & 3)));
                jc += J;
            }
        }
    }
out:
    // make sure no MMA is still running when the CTA tears down its TMEM
    tc_commit(smem_u32(S.mma_done));
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(smem_u32(S.mma_done), 0)) {
        if (globaltimer_ns() - t0 > kWaitLimitNs) break;
    }
}

template <int PASS>
__device__ void epilogue(const Params& P, const Smem& S, uint32_t tmem_base, int it0, int it1) {
    volatile int* abort_flag = S.abort_flag;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int et = threadIdx.x - 64;            // 0..255
    const int wg = (warp - 2) >> 2;             // column half
    const int q = warp & 3;                     // TMEM lane quarter this warp may access
    const int rl = q * 32 + lane;               // row (pass 1) or key (pass 2) inside a 128-tile
    const uint32_t tl = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + wg * 64;
    const float a = P.a;
    const int J = P.J;
    uint32_t jc = 0;
    int prev_unit = -1;
    uint32_t tile_par = 0;
    float m[kMaxJ], l[kMaxJ];

    for (int it = it0; it < it1; ++it) {
        const ItemInfo I = item_info(P, it);
        const int ne = min(P.n, I.N);
        const int row0 = I.slab * P.slab_rows;   // first global query row of this slab
        if (PASS == 2 && I.unit != prev_unit) {
            named_bar_sync(1, 256);
            for (int i = et; i < P.slab_rows; i += 256) S.cvec[i] = __ldcg(P.cvec + (size_t)I.unit * P.slab_rows + i);
            named_bar_sync(1, 256);
        }
        prev_unit = I.unit;
        if (PASS == 1) {
#pragma unroll
            for (int j = 0; j < kMaxJ; ++j) {
                m[j] = -INFINITY;
                l[j] = 0.f;
            }
        }
        for (int kt = I.tb; kt < I.te; ++kt) {
            float acc = 0.f;
#pragma unroll
            for (int j = 0; j < kMaxJ; ++j) {
                if (j >= J) break;
                const uint32_t buf = jc & 3;
                // after an abort every wait fails fast; the warp then skips the TMEM read (warp-uniformly,
                // tcgen05.ld is .sync.aligned) but keeps walking the same loop so the named barriers match
                const bool ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(S.tfull + buf), (jc >> 2) & 1, abort_flag));
                tc_fence_after();
                uint32_t v[64];
                if (ok) {
                    tmem_ld64(tl + buf * 128, v);
                } else {
#pragma unroll
                    for (int c = 0; c < 64; ++c) v[c] = 0u;
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(S.tempty + buf));
                ++jc;
                if (PASS == 1) {
                    // thread = query row (row0 + 128 j + rl); columns = keys kt*128 + 64 wg + c
                    const int qg = row0 + j * 128 + rl;
                    const int pos = I.N - P.n + (qg % P.n);      // local position of this query
                    if (qg < P.rows_total && pos >= 0) {
                        const int key0 = kt * kTileKeys + wg * 64;
                        const int lim = pos - key0;              // columns c <= lim are visible
                        float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
                        if (lim >= 63) {
#pragma unroll
                            for (int c = 0; c < 64; c += 4) {
                                mx0 = fmaxf(mx0, __uint_as_float(v[c]));
                                mx1 = fmaxf(mx1, __uint_as_float(v[c + 1]));
                                mx2 = fmaxf(mx2, __uint_as_float(v[c + 2]));
                                mx3 = fmaxf(mx3, __uint_as_float(v[c + 3]));
                            }
                        } else {
#pragma unroll
                            for (int c = 0; c < 64; ++c)
                                if (c <= lim) mx0 = fmaxf(mx0, __uint_as_float(v[c]));
                        }
                        const float mx = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3));
                        if (mx > -INFINITY) {
                            const float mn = fmaxf(m[j], mx * a);
                            float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
                            if (lim >= 63) {
#pragma unroll
                                for (int c = 0; c < 64; c += 4) {
                                    s0 += ex2(fmaf(__uint_as_float(v[c]), a, -mn));
                                    s1 += ex2(fmaf(__uint_as_float(v[c + 1]), a, -mn));
                                    s2 += ex2(fmaf(__uint_as_float(v[c + 2]), a, -mn));
                                    s3 += ex2(fmaf(__uint_as_float(v[c + 3]), a, -mn));
                                }
                            } else {
#pragma unroll
                                for (int c = 0; c < 64; ++c)
                                    if (c <= lim) s0 += ex2(fmaf(__uint_as_float(v[c]), a, -mn));
                            }
                            l[j] = l[j] * ex2(m[j] - mn) + ((s0 + s1) + (s2 + s3));
                            m[j] = mn;
                        }
                    }
                } else {
                    // thread = key i (kt*128 + rl); columns = query rows 128 j + 64 wg + c of the slab
                    const int i = kt * kTileKeys + rl;
                    const float4* cv = reinterpret_cast<const float4*>(S.cvec + j * 128 + wg * 64);
                    float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
                    if (kt * kTileKeys + kTileKeys - 1 <= I.N - ne) {
                        // every key of the tile is visible to every window row; rows that are not
                        // window rows carry c = +inf and contribute 2^-inf = 0
#pragma unroll
                        for (int c4 = 0; c4 < 16; ++c4) {
                            const float4 cc = cv[c4];
                            s0 += ex2(fmaf(__uint_as_float(v[4 * c4 + 0]), a, -cc.x));
                            s1 += ex2(fmaf(__uint_as_float(v[4 * c4 + 1]), a, -cc.y));
                            s2 += ex2(fmaf(__uint_as_float(v[4 * c4 + 2]), a, -cc.z));
                            s3 += ex2(fmaf(__uint_as_float(v[4 * c4 + 3]), a, -cc.w));
                        }
                    } else if (i < I.N) {
                        const int qbase = row0 + j * 128 + wg * 64;
#pragma unroll
                        for (int c4 = 0; c4 < 16; ++c4) {
                            const float4 cc = cv[c4];
                            const float cw[4] = {cc.x, cc.y, cc.z, cc.w};
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const int qg = qbase + 4 * c4 + e;
                                const int pos = I.N - P.n + (qg % P.n);
                                const bool vis = qg < P.rows_total && pos >= 0 && i <= pos;
                                const float p = ex2(fmaf(__uint_as_float(v[4 * c4 + e]), a, -cw[e]));
                                s0 += vis ? p : 0.f;
                            }
                        }
                    }
                    acc += (s0 + s1) + (s2 + s3);
                }
            }
            if (PASS == 2) {
                // combine the two column halves, then reduce over G consecutive keys (fixed order)
                float* xb = reinterpret_cast<float*>(S.xchg) + (tile_par & 1) * 128;
                float* wsum = reinterpret_cast<float*>(S.xchg) + 256 + (tile_par & 1) * 4;
                if (wg == 1) xb[rl] = acc;
                named_bar_sync(1, 256);
                if (wg == 0) {
                    const float tot = acc + xb[rl];
                    const int i = kt * kTileKeys + rl;
                    if (P.tok != nullptr && i < I.N) P.tok[(size_t)I.kk * P.T + I.base + i] = tot;
                    const int nb = (I.N + P.G - 1) / P.G;
                    const int cb = P.cb[I.r];
                    float* dst = P.blk + (size_t)I.kk * P.nb_cap + cb;
                    float s = tot;
                    const int gw = P.G < 32 ? P.G : 32;
                    for (int o = gw >> 1; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
                    if (P.G <= 32) {
                        const int g = i / P.G;
                        if ((lane & (P.G - 1)) == 0 && g < nb) dst[g] = s;
                    } else {
                        if (lane == 0) wsum[q] = s;
                        named_bar_sync(2, 128);
                        if (lane == 0) {
                            if (P.G == 64 && (q & 1) == 0) {
                                const int g = i / 64;
                                if (g < nb) dst[g] = wsum[q] + wsum[q + 1];
                            } else if (P.G == 128 && q == 0) {
                                const int g = i / 128;
                                if (g < nb) dst[g] = (wsum[0] + wsum[1]) + (wsum[2] + wsum[3]);
                            }
                        }
                    }
                }
                ++tile_par;
            }
        }
        if (PASS == 1) {
            // merge the two column halves per row, write this item's partial (m, l)
            float2* xm = reinterpret_cast<float2*>(S.xchg);
            if (wg == 1) {
#pragma unroll
                for (int j = 0; j < kMaxJ; ++j)
                    if (j < J) xm[j * 128 + rl] = make_float2(m[j], l[j]);
            }
            named_bar_sync(1, 256);
            if (wg == 0) {
#pragma unroll
                for (int j = 0; j < kMaxJ; ++j) {
                    if (j < J) {
                        const float2 o = xm[j * 128 + rl];
                        const float mm = fmaxf(m[j], o.x);
                        const float ll = mm == -INFINITY ? 0.f : l[j] * ex2(m[j] - mm) + o.y * ex2(o.x - mm);
                        P.ml[(size_t)it * P.slab_rows + j * 128 + rl] = make_float2(mm, ll);
                    }
                }
            }
            __threadfence();
            named_bar_sync(1, 256);
            if (et == 0) {
                const int2 ui = P.unit_items[I.unit];
                const int prev = atomicAdd(P.unit_done + I.unit, 1);
                *S.last_flag = (prev == ui.y - 1);
            }
            named_bar_sync(1, 256);
            if (*S.last_flag) {
                // last finisher of the unit: fold the partials in item order into c = m + log2(l)
                __threadfence();
                const int2 ui = P.unit_items[I.unit];
                for (int row = et; row < P.slab_rows; row += 256) {
                    float mm = -INFINITY;
                    for (int p = 0; p < ui.y; ++p) mm = fmaxf(mm, __ldcg(&P.ml[(size_t)(ui.x + p) * P.slab_rows + row].x));
                    float ll = 0.f;
                    if (mm > -INFINITY) {
                        for (int p = 0; p < ui.y; ++p) {
                            const float2 e = __ldcg(&P.ml[(size_t)(ui.x + p) * P.slab_rows + row]);
                            ll += e.y * ex2(e.x - mm);
                        }
                    }
                    P.cvec[(size_t)I.unit * P.slab_rows + row] = mm == -INFINITY ? INFINITY : mm + log2f(ll);
                }
            }
            named_bar_sync(1, 256);
        }
    }
}

template <int PASS, int NC>
__global__ void __launch_bounds__(kThreads, 1)
    score_pass_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK, Params P) {
    extern __shared__ uint8_t smem_raw[];
    const Smem S = carve(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(S.full + s), 1);
            mbar_init(smem_u32(S.empty + s), 1);
        }
        for (int b = 0; b < 4; ++b) {
            mbar_init(smem_u32(S.tfull + b), 1);
            mbar_init(smem_u32(S.tempty + b), 8);      // one arrival per epilogue warp
        }
        mbar_init(smem_u32(S.slab_full), 1);
        mbar_init(smem_u32(S.slab_free), 1);
        mbar_init(smem_u32(S.mma_done), 1);
        *S.abort_flag = 0;
        *S.last_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmQ);
        prefetch_tmap(&tmK);
    }
    // query rows that no TMA load ever writes (slab padding) must be finite: zero the slab once
    for (int i = threadIdx.x; i < kSlabBytes / 16; i += kThreads) reinterpret_cast<uint4*>(S.slab)[i] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
    if (warp == 1) {
        tmem_alloc(smem_u32(S.tmem_holder), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *S.tmem_holder;

    const int n_items = __ldcg(P.n_items);
    const int it0 = static_cast<int>((int64_t)blockIdx.x * n_items / gridDim.x);
    const int it1 = static_cast<int>((int64_t)(blockIdx.x + 1) * n_items / gridDim.x);

    if (warp == 0) {
        if (lane == 0) producer<NC>(P, S, &tmQ, &tmK, it0, it1);
    } else if (warp == 1) {
        if (lane == 0) mma_issuer<PASS, NC>(P, S, tmem_base, it0, it1);
    } else {
        epilogue<PASS>(P, S, tmem_base, it0, it1);
    }

    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0 && *S.abort_flag) set_status(P.status, UP_DEV_WAIT_TIMEOUT);
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

// ------------------------------------------------------------------------------------------------
// finalize: sum the per-unit partials in a fixed order and apply 1/(n_eff * Hq * G)

__device__ __forceinline__ int find_segment(const int32_t* cuts, int R, int x) {   // cuts[r] <= x < cuts[r+1]
    int lo = 0, hi = R;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (cuts[mid] <= x) lo = mid; else hi = mid;
    }
    return lo;
}

__global__ void finalize_kernel(Params P) {
    if (__ldcg(P.n_items + 1) == 0) return;   // plan rejected the varlen metadata
    const int units = P.units_per_req;
    const int nb_total = P.cb[P.R];
    const int stride = gridDim.x * blockDim.x;
    for (int gb = blockIdx.x * blockDim.x + threadIdx.x; gb < nb_total; gb += stride) {
        const int r = find_segment(P.cb, P.R, gb);
        const int ne = min(P.n, P.cu[r + 1] - P.cu[r]);
        float s = 0.f;
        for (int kk = 0; kk < units; ++kk) s += P.blk[(size_t)kk * P.nb_cap + gb];
        P.block_scores[gb] = s * (1.0f / (static_cast<float>(ne) * P.Hq * P.G));
    }
    if (P.token_scores != nullptr) {
        for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < P.T; t += stride) {
            const int r = find_segment(P.cu, P.R, t);
            const int ne = min(P.n, P.cu[r + 1] - P.cu[r]);
            float s = 0.f;
            for (int kk = 0; kk < units; ++kk) s += P.tok[(size_t)kk * P.T + t];
            P.token_scores[t] = s * (1.0f / (static_cast<float>(ne) * P.Hq));
        }
    }
}

// ------------------------------------------------------------------------------------------------
// host

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// [T, heads, dk] bf16 viewed as a 3-D tensor (dk, heads, T); box = (64, 1, rows), 128-byte swizzle
static bool make_map(CUtensorMap* m, const void* ptr, int64_t T, int heads, int dk, int rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)dk, (cuuint64_t)heads, (cuuint64_t)T};
    cuuint64_t strides[2] = {(cuuint64_t)dk * 2, (cuuint64_t)heads * dk * 2};
    cuuint32_t box[3] = {64, 1, (cuuint32_t)rows};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int PASS, int NC>
static cudaError_t launch_pass(const CUtensorMap& q, const CUtensorMap& k, const Params& P, int grid,
                               cudaStream_t st) {
    static std::once_flag once;
    static cudaError_t attr = cudaSuccess;
    std::call_once(once, [] {
        attr = cudaFuncSetAttribute(score_pass_kernel<PASS, NC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    kSmemBytes);
    });
    if (attr != cudaSuccess) return attr;
    score_pass_kernel<PASS, NC><<<grid, kThreads, kSmemBytes, st>>>(q, k, P);
    count_launch();
    return cudaGetLastError();
}

template <int NC>
static cudaError_t launch_both(const CUtensorMap& q, const CUtensorMap& k, const Params& P, int grid,
                               cudaStream_t st) {
    cudaError_t e = launch_pass<1, NC>(q, k, P, grid, st);
    if (e != cudaSuccess) return e;
    return launch_pass<2, NC>(q, k, P, grid, st);
}

}  // namespace score
}  // namespace up

using namespace up;
using namespace up::score;

extern "C" int64_t up_max_blocks(int R, int64_t T, int G) {
    if (R <= 0 || T < 0 || G <= 0) return 0;
    return T / G + R;
}

extern "C" size_t up_score_workspace_bytes(int R, int64_t T, int Hq, int Hkv, int dk, int G, int n, int64_t nb_cap,
                                           int with_token_scores) {
    Geometry g;
    if (R <= 0 || T < 0 || T >= (int64_t(1) << 31) || nb_cap < 0 || !geometry(Hq, Hkv, dk, n, &g)) return 0;
    (void)G;
    return layout(R, T, g, Hkv, nb_cap, with_token_scores != 0).total;
}

extern "C" up_status up_score_blocks(const uint16_t* Q, const uint16_t* K, const int32_t* cu_seqlens, int R,
                                     int64_t T, int Hq, int Hkv, int dk, int G, int n, float sm_scale,
                                     const int32_t* cu_blocks, int64_t nb_cap, float* block_scores,
                                     float* token_scores, void* ws, size_t ws_bytes, int32_t* dev_status,
                                     void* stream) {
    if (!Q || !K || !cu_seqlens || !cu_blocks || !block_scores || !ws || !dev_status) return UP_ERR_ARG;
    if (R <= 0 || T < 0 || T >= (int64_t(1) << 31) || nb_cap < 0 || !(sm_scale > 0.f) || !isfinite(sm_scale))
        return UP_ERR_ARG;
    Geometry g;
    if (!geometry(Hq, Hkv, dk, n, &g)) return UP_ERR_SHAPE;
    if (G != 16 && G != 32 && G != 64 && G != 128) return UP_ERR_SHAPE;
    if (!aligned16(Q) || !aligned16(K) || !aligned16(ws)) return UP_ERR_SHAPE;
    const Layout L = layout(R, T, g, Hkv, nb_cap, token_scores != nullptr);
    if (ws_bytes < L.total) return UP_ERR_WORKSPACE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    uint8_t* w = static_cast<uint8_t*>(ws);
    Params P{};
    P.cu = cu_seqlens;
    P.cb = cu_blocks;
    P.R = R;
    P.T = static_cast<int>(T);
    P.Hq = Hq;
    P.Hkv = Hkv;
    P.dk = dk;
    P.G = G;
    P.n = n;
    P.group = g.group;
    P.rows_total = g.rows_total;
    P.slab_rows = g.slab_rows;
    P.slabs = g.slabs;
    P.J = g.J;
    P.box_rows = g.box_rows;
    P.units_per_req = Hkv * g.slabs;
    P.a = sm_scale * 1.4426950408889634f;
    P.nb_cap = nb_cap;
    P.items = reinterpret_cast<int4*>(w + L.items);
    P.unit_items = reinterpret_cast<int2*>(w + L.unit_items);
    P.n_items = reinterpret_cast<int*>(w + L.n_items);
    P.unit_done = reinterpret_cast<int*>(w + L.unit_done);
    P.ml = reinterpret_cast<float2*>(w + L.ml);
    P.cvec = reinterpret_cast<float*>(w + L.cvec);
    P.blk = reinterpret_cast<float*>(w + L.blk);
    P.tok = token_scores ? reinterpret_cast<float*>(w + L.tok) : nullptr;
    P.block_scores = block_scores;
    P.token_scores = token_scores;
    P.status = dev_status;

    plan_kernel<<<1, 1024, 0, st>>>(P);
    count_launch();
    if (cudaGetLastError() != cudaSuccess) return UP_ERR_CUDA;
    if (T > 0) {
        CUtensorMap tq, tk;
        if (!make_map(&tq, Q, T, Hq, dk, g.box_rows) || !make_map(&tk, K, T, Hkv, dk, kTileKeys)) return UP_ERR_CUDA;
        const int grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(num_sms(), L.items_cap)));
        cudaError_t e;
        switch (g.nc) {
            case 1: e = launch_both<1>(tq, tk, P, grid, st); break;
            case 2: e = launch_both<2>(tq, tk, P, grid, st); break;
            default: e = launch_both<4>(tq, tk, P, grid, st); break;
        }
        if (e != cudaSuccess) return UP_ERR_CUDA;
    }
    const int fgrid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(4 * num_sms(), cdiv(std::max<int64_t>(nb_cap, T), 256))));
    finalize_kernel<<<fgrid, 256, 0, st>>>(P);
    count_launch();
    return cudaGetLastError() == cudaSuccess ? UP_OK : UP_ERR_CUDA;
}
