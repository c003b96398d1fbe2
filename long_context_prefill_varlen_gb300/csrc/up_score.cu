// up_score_blocks: block-level importance of UniPrefill ("UniPrefill: Universal Long-Context
// Prefill Acceleration via Block-wise Dynamic Sparsification", arXiv 2605.06221, section 3.2,
// Eqs. 2-4, and the kernel pipeline of section 3.5, Eq. 13).
//
// For every request r, KV head kh and the group x n window query rows that read kh, S = Qwin . K^T
// is computed on tcgen05 (query rows in TMEM lanes, 128 keys per tile in columns) in one of two ways.
//   one pass (the default)  per row the online max m and sum l of 2^(S*a - m) over the causal key
//           range, per work item (kItemTiles key tiles) a partial (m, l), and per key tile the sums of
//           2^(S*a - m_t) over each block with their reference maxima m_t; the merge kernel folds the
//           partials into c = m + log2(l) per row, and the reduce kernel forms b_g from the block sums
//           scaled by 2^(m_t - c) (see the one-pass section).  S is computed once and never stored.
//   two passes (when per-token scores are asked for)  pass 1 as above without the block sums, the
//           merge, then pass 2 recomputes S^T = K . Qwin^T (keys in TMEM lanes) and sums
//           P = 2^(S*a - c_row) per key over its rows, reduced over G keys with warp shuffles into
//           per-(unit, block) partials; the final kernel divides by n_eff * Hq * G.
// a = sm_scale * log2(e): the softmax is computed in base 2, exactly equal to exp in base e.
//
// CTA layout (608 threads, one CTA per SM, persistent over a contiguous range of work items):
//   warp 0     TMA producer: the query slab of the current unit, then K tiles into a 5-stage ring
//   warps 1, 18  tcgen05.mma issuers (warp 1 also allocates TMEM; each runs its loop on the whole warp
//              and issues from one elected lane), see mma_issuer
//   warps 2-17 four epilogue warpgroups.  A job is one 128 x W fp32 accumulator (W = 128 query rows;
//              W = 256 in pass 2 when the slab has 256 rows).  One pass: warpgroup w drains TMEM
//              buffer w whole at d_k <= 128, and at d_k = 256 the pairs of warpgroups drain alternate
//              buffers, 64 columns each.  Two passes: with J jobs per key tile warpgroup g takes jobs
//              g, g+4, ... when J >= 3, half a job when J = 2 and a quarter when J = 1.  TMEM is read
//              in 16- or 32-column chunks, the next chunk's load in flight while the current one is
//              reduced.
// TMEM: the whole 512 columns, a ring of 4 (W = 128) or 2 (W = 256) accumulators.
// Per element the epilogue spends one ex2 on the SFU (32/clk/SM on this part, the same rate at
// which the tensor core produces S elements at d_k = 128) plus one FFMA and one FADD.
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
constexpr int kEpiThreads = 512;
constexpr int kIssuers = 2;                     // MMA issuer warps (warps 1 and 18); see mma_issuer
constexpr int kEpiWarp0 = 2;                    // epilogue warps 2..17
constexpr int kIssuer1Warp = kEpiWarp0 + kEpiThreads / 32;
constexpr int kThreads = 64 + kEpiThreads + 32 * (kIssuers - 1);
constexpr int kMaxJ = 8;                        // 128-row jobs per slab (d_k = 64 -> 8)
constexpr int kTmemCols = 512;
constexpr uint32_t kIdesc = idesc_bf16_f32(128, 128);
constexpr uint32_t kIdescWide = idesc_bf16_f32(128, 256);
constexpr int kCtrlBytes = 256;
constexpr int kCvecFloats = 2048;               // pass 2: row normalisers; one pass (d_k = 256): half exchange
constexpr int kXchgBytes = 4 * 2 * 128 * 8;     // pass 1: (m,l) of 4 warpgroups x 2 jobs
constexpr int kSmemBytes = 1024 + kSlabBytes + kStages * kStageBytes + kCtrlBytes + kCvecFloats * 4 + kXchgBytes;

struct Geometry {
    int group, rows_total, slab_rows, slabs, J, box_rows, nc;
};

struct Layout {
    size_t items, unit_items, n_items, ml, cvec, blk, tok, be, bm, total;
    int64_t items_cap, units;
};

struct Params {
    const int32_t* cu;
    const int32_t* cb;
    int R, T, Hq, Hkv, dk, G, n, group, rows_total, slab_rows, slabs, J, box_rows, units_per_req;
    int wide2;             // pass 2 takes one 256-row job per key tile (J = 2)
    int nsets;             // CTA sets that walk the same key tiles side by side (see plan)
    float a;
    int64_t nb_cap;
    int4* items;
    int2* unit_items;
    int* n_items;
    float2* ml;
    float* cvec;
    float* blk;
    float* tok;
    float* be;             // one pass: per (unit, key tile, block of the tile, row) block sums of 2^(S*a - m_t)
    float* bm;             // one pass: per (unit, key tile, row) the reference m_t of those sums
    int spt;               // one pass: blocks per key tile (128 / G)
    // element counts of the workspace arrays (checked by the bounds-checked build)
    int64_t lim_items, lim_units, lim_ml, lim_cvec, lim_blk, lim_tok, lim_be, lim_bm;
    float* block_scores;
    float* token_scores;
    int32_t* status;
};

// Jobs of one key tile in a pass: J jobs of W query rows (one 128 x W fp32 accumulator each, W TMEM
// columns) in a ring of nbuf = 512 / W TMEM buffers, wpj warpgroups draining each job (W / wpj
// columns each).  Pass 1 keeps W = 128 (a query row per TMEM lane).  Pass 2 puts keys in the lanes,
// and with a 256-row slab (J = 2: d_k = 256, or 256 window rows per KV head) it takes one job of
// W = 256 per tile, drained by all four warpgroups: a 128 x 256 x 16 MMA reads 12 KB of shared
// memory in 128 cycles (96 B per clock), where two 128 x 128 x 16 MMAs read 16 KB, the whole 128 B
// per clock, and the TMA writes of the K tiles wait for gaps.  Measured on the score call: 7-8%
// faster at d_k = 256; with the 512-row slab of d_k = 128 (two 256-row jobs) 1-4% slower than four
// 128-row jobs, whose TMEM buffers come free sooner, so J = 4 keeps W = 128.
struct JobMap {
    int J, W, nbuf, nb_log, wpj;
};
__host__ __device__ constexpr int wg_per_job(int J) { return J == 1 ? 4 : J == 2 ? 2 : 1; }
// PASS 3 is the one-pass form of pass 1 (epilogue_one_pass_whole / _pairs): the jobs of pass 1, each
// TMEM buffer drained by one warpgroup, or at d_k = 256 by a pair of warpgroups (64 columns each).
template <int PASS>
__host__ __device__ __forceinline__ JobMap job_map(const Params& P) {
    if (PASS == 2 && P.wide2) return JobMap{P.J / 2, 256, 2, 1, 4};
    if (PASS == 3) return JobMap{P.J, 128, 4, 2, 1};
    return JobMap{P.J, 128, 4, 2, wg_per_job(P.J)};
}

// The one pass applies to slabs of 1, 2 or 4 jobs (a warpgroup then always drains the same job).
__host__ __device__ constexpr bool one_pass_ok(int J) { return J == 1 || J == 2 || J == 4; }
// Sub-block sums per half-tile (64 keys) of the one pass: the blocks of G <= 64 keys in it, or one.
__host__ __device__ constexpr int sub_blocks_per_half(int G) { return G >= 64 ? 1 : 64 / G; }


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

// CTA sets of the score passes: every unit of a request (KV heads x slabs) when that many sets leave
// at most 2% of the SMs idle, else the slabs of a KV head under the same rule, else one set.
static int work_sets(int units_per_req, int slabs, int sms) {
    auto fits = [&](int s) { return s <= sms && (sms % s) * 50 <= sms; };
    if (units_per_req > 1 && fits(units_per_req)) return units_per_req;
    if (slabs > 1 && fits(slabs)) return slabs;
    return 1;
}

static Layout layout(int R, int64_t T, const Geometry& g, int Hkv, int64_t nb_cap, bool tok, int G) {
    Layout L{};
    L.items_cap = (cdiv(T, (int64_t)kTileKeys * kItemTiles) + R) * Hkv * g.slabs;
    L.units = (int64_t)R * Hkv * g.slabs;
    size_t o = 0;
    auto take = [&](size_t bytes) { size_t at = o; o = align_up(o + bytes, 256); return at; };
    L.items = take(sizeof(int4) * 2 * L.items_cap);      // two entries per item (see item_decode)
    L.unit_items = take(sizeof(int2) * L.units);
    L.n_items = take(16);
    L.ml = take(sizeof(float2) * L.items_cap * g.slab_rows);
    L.cvec = take(sizeof(float) * L.units * g.slab_rows);
    L.blk = take(sizeof(float) * (size_t)Hkv * g.slabs * 4 * nb_cap);      // one partial per warpgroup
    L.tok = tok ? take(sizeof(float) * (size_t)Hkv * g.slabs * 4 * T) : 0;
    if (one_pass_ok(g.J)) {
        // block sums and their reference maxima of the one pass, per (unit, key tile, row); a unit's tiles
        // start at twice its first item's index in the plan's dense per-unit item numbering
        const size_t tiles = static_cast<size_t>(L.items_cap) * kItemTiles;
        L.be = take(sizeof(float) * tiles * (kTileKeys / G) * g.slab_rows);
        L.bm = take(sizeof(float) * tiles * g.slab_rows);
    }
    L.total = o;
    return L;
}

// ------------------------------------------------------------------------------------------------
// plan: validate the varlen metadata and lay out the work items (one CTA)

// exclusive prefix sum over the CTA (blockDim.x a multiple of 32, at most 1024); sh holds 32 ints
__device__ __forceinline__ int block_exclusive_scan(int v, int* sh, int* total) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) sh[w] = x;
    __syncthreads();
    if (w == 0) {
        int s = lane < nw ? sh[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o) s += y;
        }
        sh[lane] = s;   // inclusive over warps (warps past the last add 0)
    }
    __syncthreads();
    const int before = (w > 0 ? sh[w - 1] : 0) + x - v;
    *total = sh[31];
    __syncthreads();
    return before;
}

// Up to this many requests every plan CTA keeps each request's first run-0 item in shared memory and
// the item list is written by a grid of CTAs; beyond it one CTA writes the list (searching the
// unit offsets in global memory).
constexpr int kPlanThreads = 1024;
constexpr int kPlanSmemReqs = 4096;
constexpr int kPlanScratch = (kPlanSmemReqs + 64) * 4;   // bytes of the query slab a planning pass borrows

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(Params P) {
    pdl_wait();
    pdl_trigger();
    __shared__ int s_bad;
    __shared__ int s_scan[32];
    __shared__ int s_first[kPlanSmemReqs];
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
        if (tid == 0 && blockIdx.x == 0) {
            set_status(P.status, (s_bad & 1) ? UP_DEV_BAD_CU_SEQLENS : UP_DEV_BAD_CU_BLOCKS);
            P.n_items[0] = 0;
            P.n_items[1] = 0;      // metadata invalid: finalize writes nothing
        }
        return;
    }
    const int NS = P.nsets;
    const bool in_smem = P.R <= kPlanSmemReqs;
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
    int off = block_exclusive_scan(local, s_scan, &total);
    for (int r = r0; r < r1; ++r) {
        const int ni = nitems(r);
        if (blockIdx.x == 0) {
            for (int kk = 0; kk < P.units_per_req; ++kk) {
                const int u = r * P.units_per_req + kk;
                if (UP_IN(u, P.lim_units, P.status)) P.unit_items[u] = make_int2(off + kk * ni, ni);
            }
        }
        if (in_smem) s_first[r] = off / NS;
        off += ni * P.units_per_req;
    }
    __syncthreads();
    // Items are listed set-major.  Unit kk of a request (KV head kh, query slab sl, kk = kh * slabs +
    // sl) belongs to set kk % nsets; the list holds all items of set 0 in (request, kk / nsets, tile
    // pair) order, then the same sequence for set 1, and so on.  Every (request, tile pair) has an
    // item in each unit, so the nsets runs are equally long and item s * run + i is item i of run 0
    // moved to set s.  The score passes split every run identically over nsets sets of CTAs, so the
    // CTAs holding the units of one request walk the same key tiles side by side: with nsets = slabs
    // a K tile is read from DRAM about once instead of once per slab, and with nsets = Hkv * slabs the
    // KV heads of a token range are also read together (whole rows of the [T, Hkv, d_k] K tensor).
    // A unit's items are therefore not contiguous in the list; its pass-1 partials are indexed by the
    // item's tile pair inside the unit (unit_items[u].x + pair).  nsets = 1 is the plain order.
    const int run = total / NS;
    auto first = [&](int r) { return in_smem ? s_first[r] : P.unit_items[r * P.units_per_req].x / NS; };
    for (int it = blockIdx.x * blockDim.x + tid; it < total; it += gridDim.x * blockDim.x) {
        const int set = it / run, rel = it - set * run;
        // the request: the largest r whose first run-0 item (its first item / NS) is <= rel; never an
        // empty request (an empty request shares its first item with the next one, and rel < run
        // excludes an empty last request)
        int lo = 0, hi = P.R;
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (first(mid) <= rel) lo = mid; else hi = mid;
        }
        const int r = lo;
        const int ni = nitems(r);
        const int rel2 = rel - first(r);
        const int kq = rel2 / ni, sidx = rel2 % ni;
        const int kk = kq * NS + set;
        const int N = P.cu[r + 1] - P.cu[r];
        const int ntiles = (N + kTileKeys - 1) / kTileKeys;
        if (UP_IN(it, P.lim_items, P.status)) {
            P.items[2 * it] = make_int4(r, kk, sidx * kItemTiles, min(ntiles, (sidx + 1) * kItemTiles));
            P.items[2 * it + 1] = make_int4(P.cu[r], N, first(r) * NS + kk * ni, ni);
        }
    }
    if (tid == 0 && blockIdx.x == 0) {
        P.n_items[0] = total;
        P.n_items[1] = 1;          // metadata validated
    }
}

// Up to kPlanSmemReqs requests the one pass plans inside its own launch (no plan kernel before it):
// every CTA validates the metadata, scans the requests' item counts into shared memory and writes the
// entries of its own items [it0, it1) and the unit offsets of the requests r with
// r mod gridDim.x == blockIdx.x (read by the merge and reduce kernels); CTA 0 writes the item count.
// The list and the split over the CTAs are those of plan_kernel.  False when the metadata is invalid
// (CTA 0 records the status; every CTA returns false and does no work).  All threads call it; s_first
// holds kPlanSmemReqs ints and s_red 33.
__device__ bool plan_prologue(const Params& P, int* s_first, int* s_red, int& it0, int& it1) {
    const int tid = threadIdx.x, nt = blockDim.x;
    if (tid == 0) s_red[32] = 0;
    __syncthreads();
    for (int r = tid; r < P.R; r += nt) {
        const int c0 = P.cu[r], c1 = P.cu[r + 1];
        if ((r == 0 && c0 != 0) || c1 < c0 || c1 > P.T || (r == P.R - 1 && c1 != P.T)) atomicOr(&s_red[32], 1);
        const int nb = (c1 - c0 + P.G - 1) / P.G;
        const int b0 = P.cb[r], b1 = P.cb[r + 1];
        if ((r == 0 && b0 != 0) || b1 - b0 != nb || (int64_t)b1 > P.nb_cap) atomicOr(&s_red[32], 2);
    }
    __syncthreads();
    const int bad = s_red[32];
    if (bad) {
        if (tid == 0 && blockIdx.x == 0) {
            set_status(P.status, (bad & 1) ? UP_DEV_BAD_CU_SEQLENS : UP_DEV_BAD_CU_BLOCKS);
            P.n_items[0] = 0;
            P.n_items[1] = 0;
        }
        it0 = it1 = 0;
        return false;
    }
    const int NS = P.nsets, upr = P.units_per_req;
    auto nitems = [&](int r) {
        const int N = P.cu[r + 1] - P.cu[r];
        return ((N + kTileKeys - 1) / kTileKeys + kItemTiles - 1) / kItemTiles;
    };
    const int per = (P.R + nt - 1) / nt;
    const int r0 = min(P.R, tid * per), r1 = min(P.R, r0 + per);
    int local = 0;
    for (int r = r0; r < r1; ++r) local += nitems(r) * upr;
    int total = 0;
    int off = block_exclusive_scan(local, s_red, &total);
    for (int r = r0; r < r1; ++r) {
        const int ni = nitems(r);
        if (r % gridDim.x == blockIdx.x)
            for (int kk = 0; kk < upr; ++kk) {
                const int u = r * upr + kk;
                if (UP_IN(u, P.lim_units, P.status)) P.unit_items[u] = make_int2(off + kk * ni, ni);
            }
        s_first[r] = off / NS;
        off += ni * upr;
    }
    if (tid == 0 && blockIdx.x == 0) {
        P.n_items[0] = total;
        P.n_items[1] = 1;
    }
    __syncthreads();
    const int groups = gridDim.x / NS, run = total / NS;
    const int set = blockIdx.x / groups, g = blockIdx.x % groups;
    it0 = set * run + static_cast<int>((int64_t)g * run / groups);
    it1 = set * run + static_cast<int>((int64_t)(g + 1) * run / groups);
    for (int it = it0 + tid; it < it1; it += nt) {
        const int rel = it - set * run;
        int lo = 0, hi = P.R;
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (s_first[mid] <= rel) lo = mid; else hi = mid;
        }
        const int r = lo, ni = nitems(r);
        const int rel2 = rel - s_first[r];
        const int kq = rel2 / ni, sidx = rel2 % ni;
        const int kk = kq * NS + set;
        const int N = P.cu[r + 1] - P.cu[r];
        const int ntiles = (N + kTileKeys - 1) / kTileKeys;
        if (UP_IN(it, P.lim_items, P.status)) {
            P.items[2 * it] = make_int4(r, kk, sidx * kItemTiles, min(ntiles, (sidx + 1) * kItemTiles));
            P.items[2 * it + 1] = make_int4(P.cu[r], N, s_first[r] * NS + kk * ni, ni);
        }
    }
    return true;
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
    uint64_t* mma_done;    // [kIssuers]
    uint64_t* tok;         // [2]        turn of issuer 0 / 1 to issue its next job (jobs-outer path)
    uint32_t* tmem_holder;
    int* abort_flag;
    float* cvec;           // [kCvecFloats]
    uint8_t* xchg;         // [kXchgBytes]
};

// the barriers (full, empty, tfull, tempty, slab_full, slab_free, mma_done, tok), the TMEM address and the
// abort flag fit the control block
static_assert((2 * kStages + 8 + 2 + kIssuers + 2) * 8 + 8 <= kCtrlBytes, "control block too small");

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
    s.tok = b + 2 * kStages + 10 + kIssuers;
    s.tmem_holder = reinterpret_cast<uint32_t*>(b + 2 * kStages + 12 + kIssuers);
    s.abort_flag = reinterpret_cast<int*>(s.tmem_holder + 1);
    s.cvec = reinterpret_cast<float*>(ctrl + kCtrlBytes);
    s.xchg = reinterpret_cast<uint8_t*>(s.cvec + kCvecFloats);
    return s;
}

struct ItemInfo {
    int r, kk, tb, te, unit, base, N, kh, slab;
    int2 ui;               // the unit's first item in the per-unit numbering, and its item count
};

// Values read from memory are not known to be warp-uniform; the MMA, TMA and TMEM-load operands
// derived from them must be.  Broadcasting from lane 0 makes the uniformity explicit, so everything
// computed from the schedule below stays in warp-uniform registers (every caller is a full warp).
__device__ __forceinline__ int uni(int v) { return __shfl_sync(0xffffffffu, v, 0); }

// An item is two entries of the list: (request, unit of the request, first tile, end tile) and (the
// request's first token, its length, the unit's first item in the per-unit numbering, the unit's item
// count), loaded together (no dependent loads).  The producer and the MMA
// issuers, which set the pace, load the next item's entries while they work on the current one.
__device__ __forceinline__ void item_load(const Params& P, int it, int it1, int4& a, int4& b) {
    if (it < it1 && UP_IN(it, P.lim_items, P.status)) {
        a = P.items[2 * it];
        b = P.items[2 * it + 1];
    } else {
        a = b = make_int4(0, 0, 0, 0);
    }
}
__device__ __forceinline__ ItemInfo item_decode(const Params& P, const int4& a, const int4& b) {
    ItemInfo I;
    I.r = uni(a.x);
    I.kk = uni(a.y);
    I.tb = uni(a.z);
    I.te = uni(a.w);
    I.unit = I.r * P.units_per_req + I.kk;
    I.base = uni(b.x);
    I.N = uni(b.y);
    I.ui = make_int2(uni(b.z), uni(b.w));
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
    // the whole warp walks the schedule (warp-uniform values); one elected lane issues the copies
    volatile int* abort_flag = S.abort_flag;
    int prev_unit = -1;
    uint32_t stage_cnt = 0, slab_cnt = 0;
    const uint32_t slab_addr = smem_u32(S.slab), stage_addr = smem_u32(S.stages);
    const bool leader = elect_one();
    int4 na, nb;
    item_load(P, it0, it1, na, nb);
    for (int it = it0; it < it1; ++it) {
        const ItemInfo I = item_decode(P, na, nb);
        item_load(P, it + 1, it1, na, nb);
        if (I.unit != prev_unit) {
            if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(S.slab_free), (slab_cnt & 1) ^ 1, abort_flag))) {
                if (leader) drain_loads(S, stage_cnt, slab_cnt);
                return;
            }
            const int row0 = I.slab * P.slab_rows;
            const int rows = min(P.slab_rows, P.rows_total - row0);
            const uint32_t bar = smem_u32(S.slab_full);
            if (leader) {
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
            }
            __syncwarp();
            ++slab_cnt;
            prev_unit = I.unit;
        }
        for (int kt = I.tb; kt < I.te; ++kt) {
#pragma unroll
            for (int c = 0; c < NC; ++c) {
                const uint32_t s = stage_cnt % kStages, ph = (stage_cnt / kStages) & 1;
                if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(S.empty + s), ph ^ 1, abort_flag))) {
                    if (leader) drain_loads(S, stage_cnt, slab_cnt);
                    return;
                }
                if (leader) {
                    mbar_arrive_expect_tx(smem_u32(S.full + s), kStageBytes);
                    tma_load_3d(stage_addr + s * kStageBytes, tmK, smem_u32(S.full + s), c * 64, I.kh,
                                I.base + kt * kTileKeys);
                }
                __syncwarp();
                ++stage_cnt;
            }
        }
    }
}

// Descriptor of a K-major SW128 operand advanced by `bytes` (a multiple of 16): the start address
// occupies the low 14 bits as address >> 4 and every operand lies below 256 KB of shared memory, so
// the advance is a plain add on the descriptor.
__device__ __forceinline__ uint64_t desc_add(uint64_t d, uint32_t bytes) { return d + (bytes >> 4); }

// Two issuer warps.  A tcgen05.mma returns to its thread only once the tensor core's queue has room
// (about five 128 x 128 x 16 steps, ~320 cycles of work), so an issuer runs at most that far ahead of
// the pipe; a commit returns after ~55 cycles but holds the thread's next MMAs until the ones it tracks
// have completed (timed on this part: ~80 idle cycles per commit when no other thread's MMAs are
// queued).  Two issuers keep the queue filled across each other's commits and waits.  Issuer w
// issues the jobs q (running job count) with q mod 2 = w, i.e. those in TMEM buffers w and w + 2
// (w alone for the two 256-column buffers of a wide pass).
//   jobs outer (d_k <= 128)  the two also hand each other the turn to issue through an mbarrier after
//       each job, so the tensor core receives whole jobs in order and they complete one after
//       another, while each issuer's commit, buffer wait and loop overlap the other's MMAs.
//   chunks outer (d_k = 256)  with J = 2 each issuer has one job per key tile; per K stage both issue
//       their job's MMAs.  (A third issuer warp, the buffers handed out by b mod 3, measured 5-6% slower
//       with this epilogue; with one issuer per buffer a 21st warp would cut the registers to 80.)
// Every use of a TMEM buffer comes from the same warp in order, so its waits for the buffer always
// refer to the phase just before the current one.  A commit tracks only its own thread's MMAs, so
// every barrier that releases an operand (K stage, query slab) takes one commit from each issuer,
// and each issuer waits for a stage to land before it commits the stage's release, even when it
// issued no job on that tile: its arrival can then never count toward a later use of the stage.
static_assert(kThreads == 608 && kIssuer1Warp + kIssuers - 2 == kThreads / 32 - 1,
              "warps: producer 0, issuers 1 and 18, epilogue 2-17");
template <int PASS, int NC>
__device__ void mma_issuer(const Params& P, const Smem& S, uint32_t tmem_base, int it0, int it1, uint32_t w) {
    volatile int* abort_flag = S.abort_flag;
    int prev_unit = -1;
    uint32_t stage_cnt = 0, slab_cnt = 0, jc = 0;
    const JobMap jm = job_map<PASS>(P);
    const int J = jm.J;
    const uint32_t idesc = jm.W == 256 ? kIdescWide : kIdesc;
    // base descriptors: query slab at (chunk 0, row 0) and K stage 0; strides in bytes
    const uint64_t slab_d0 = sdesc_sw128(smem_u32(S.slab));
    const uint64_t stage_d0 = sdesc_sw128(smem_u32(S.stages));
    const uint32_t slab_chunk_bytes = static_cast<uint32_t>(P.slab_rows) * 128u;   // one 64-wide k chunk
    // the whole warp runs this loop with warp-uniform values; one elected lane issues the MMAs and
    // the commits (a commit tracks the MMAs issued by its own thread)
    const bool leader = elect_one();
    auto wait_all = [&](uint32_t bar, uint32_t parity) {
        return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag));
    };
    auto commit = [&](uint32_t bar) {
        if (leader) tc_commit(bar);
        __syncwarp();
    };
    // job q by issuer q mod 2: its buffer is b = q mod nbuf, so buffer b always by issuer b mod 2
    auto mine = [&](uint32_t q) { return (q & 1u) == w; };
    int4 na, nb;
    item_load(P, it0, it1, na, nb);
    for (int it = it0; it < it1; ++it) {
        const ItemInfo I = item_decode(P, na, nb);
        item_load(P, it + 1, it1, na, nb);
        if (I.unit != prev_unit) {
            if (prev_unit >= 0) commit(smem_u32(S.slab_free));
            if (!wait_all(smem_u32(S.slab_full), slab_cnt & 1)) goto out;
            ++slab_cnt;
            tc_fence_after();
            prev_unit = I.unit;
        }
        for (int kt = I.tb; kt < I.te; ++kt) {
            if (NC <= 2) {
                // jobs outer: the tile's K stages stay resident while the J jobs run
                bool landed = false;
                for (int j = 0; j < J; ++j) {
                    const uint32_t q = jc + j, buf = q & (jm.nbuf - 1);
                    if (!mine(q)) continue;
                    if (!wait_all(smem_u32(S.tempty + buf), ((q >> jm.nb_log) & 1) ^ 1)) goto out;
                    // this issuer's turn: the other one has issued job q - 1 (issuer 0's first job has no wait)
                    const int turn = static_cast<int>(q >> 1) - (w == 0 ? 1 : 0);
                    if (turn >= 0 && !wait_all(smem_u32(S.tok + w), turn & 1)) goto out;
                    tc_fence_after();
                    const uint64_t qd = desc_add(slab_d0, j * jm.W * 128);
                    const uint32_t d_tmem = tmem_base + buf * jm.W;
#pragma unroll
                    for (int c = 0; c < NC; ++c) {
                        const uint32_t sc = stage_cnt + c, s = sc % kStages;
                        if (!landed) {
                            if (!wait_all(smem_u32(S.full + s), (sc / kStages) & 1)) goto out;
                            tc_fence_after();
                        }
                        const uint64_t kd = desc_add(stage_d0, s * kStageBytes);
                        const uint64_t qdc = desc_add(qd, c * slab_chunk_bytes);
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const uint64_t a = PASS != 2 ? desc_add(qdc, k * 32) : desc_add(kd, k * 32);
                            const uint64_t b = PASS != 2 ? desc_add(kd, k * 32) : desc_add(qdc, k * 32);
                            if (leader) tc_mma_bf16(d_tmem, a, b, idesc, (c | k) != 0);
                        }
                    }
                    landed = true;
                    if (leader) mbar_arrive(smem_u32(S.tok + (w ^ 1u)));       // job q + 1's turn
                    __syncwarp();
                    commit(smem_u32(S.tfull + buf));
                }
#pragma unroll
                for (int c = 0; c < NC; ++c) {
                    const uint32_t sc = stage_cnt + c;
                    if (!landed && !wait_all(smem_u32(S.full + sc % kStages), (sc / kStages) & 1)) goto out;
                    commit(smem_u32(S.empty + sc % kStages));
                }
                stage_cnt += NC;
                jc += J;
            } else {
                // chunks outer (d_k = 256, J <= 2): each K stage is released as soon as all jobs used it
                for (int j = 0; j < J; ++j) {
                    const uint32_t q = jc + j;
                    if (mine(q) && !wait_all(smem_u32(S.tempty + (q & (jm.nbuf - 1))), ((q >> jm.nb_log) & 1) ^ 1))
                        goto out;
                }
                tc_fence_after();
#pragma unroll
                for (int c = 0; c < NC; ++c) {
                    const uint32_t s = stage_cnt % kStages;
                    if (!wait_all(smem_u32(S.full + s), (stage_cnt / kStages) & 1)) goto out;
                    tc_fence_after();
                    const uint64_t kd = desc_add(stage_d0, s * kStageBytes);
                    for (int j = 0; j < J; ++j) {
                        if (!mine(jc + j)) continue;
                        const uint32_t d_tmem = tmem_base + ((jc + j) & (jm.nbuf - 1)) * jm.W;
                        const uint64_t qdc = desc_add(slab_d0, j * jm.W * 128 + c * slab_chunk_bytes);
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const uint64_t a = PASS != 2 ? desc_add(qdc, k * 32) : desc_add(kd, k * 32);
                            const uint64_t b = PASS != 2 ? desc_add(kd, k * 32) : desc_add(qdc, k * 32);
                            if (leader) tc_mma_bf16(d_tmem, a, b, idesc, (c | k) != 0);
                        }
                    }
                    commit(smem_u32(S.empty + s));
                    ++stage_cnt;
                }
                for (int j = 0; j < J; ++j)
                    if (mine(jc + j)) commit(smem_u32(S.tfull + ((jc + j) & (jm.nbuf - 1))));
                jc += J;
            }
        }
    }
out:
    // make sure none of this warp's MMAs is still running when the CTA tears down its TMEM
    __syncwarp();
    commit(smem_u32(S.mma_done + w));
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(smem_u32(S.mma_done + w), 0)) {
        if (globaltimer_ns() - t0 > kWaitLimitNs) break;
    }
}

// Job map of the epilogue (one place for both the dispatch and the epilogue): with J jobs of W rows
// per key tile and wpj warpgroups on each job (job_map), each warpgroup reads W / 16 / wpj 16-column
// chunks of a job (chunks_per_slice(J) for W = 128) and warpgroup g takes the jobs
// g / wpj + u * (4 / wpj).  (Splitting J = 4 jobs of 128 rows over pairs of warpgroups, so that each
// pair alternates between two TMEM buffers, measured slower: the per-job overheads doubled.)
__host__ __device__ constexpr int chunks_per_slice(int J) { return 8 / wg_per_job(J); }
static_assert(chunks_per_slice(1) == 2 && chunks_per_slice(2) == 4 && chunks_per_slice(3) == 8 &&
                  chunks_per_slice(4) == 8 && chunks_per_slice(8) == 8,
              "a job slice must cover 128 / wg_per_job columns");

__device__ __forceinline__ float max3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// 16 consecutive fp32 columns of this warp's 32 TMEM lanes, without waiting
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
        : "r"(taddr)
        : "memory");
}
// wait for every outstanding tcgen05.ld of this thread, then pin the destination registers after
// the wait so that no use of them can be scheduled before it
__device__ __forceinline__ void tmem_wait_pin(uint32_t (&v)[16]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
    asm volatile(""
                 : "+r"(v[0]), "+r"(v[1]), "+r"(v[2]), "+r"(v[3]), "+r"(v[4]), "+r"(v[5]), "+r"(v[6]), "+r"(v[7]),
                   "+r"(v[8]), "+r"(v[9]), "+r"(v[10]), "+r"(v[11]), "+r"(v[12]), "+r"(v[13]), "+r"(v[14]),
                   "+r"(v[15]));
}

// 32 consecutive fp32 columns of this warp's 32 TMEM lanes, without waiting
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
          "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
          "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_wait_pin32(uint32_t (&v)[32]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
    asm volatile(""
                 : "+r"(v[0]), "+r"(v[1]), "+r"(v[2]), "+r"(v[3]), "+r"(v[4]), "+r"(v[5]), "+r"(v[6]), "+r"(v[7]),
                   "+r"(v[8]), "+r"(v[9]), "+r"(v[10]), "+r"(v[11]), "+r"(v[12]), "+r"(v[13]), "+r"(v[14]),
                   "+r"(v[15]));
    asm volatile(""
                 : "+r"(v[16]), "+r"(v[17]), "+r"(v[18]), "+r"(v[19]), "+r"(v[20]), "+r"(v[21]), "+r"(v[22]),
                   "+r"(v[23]), "+r"(v[24]), "+r"(v[25]), "+r"(v[26]), "+r"(v[27]), "+r"(v[28]), "+r"(v[29]),
                   "+r"(v[30]), "+r"(v[31]));
}

__device__ __forceinline__ float f(uint32_t x) { return __uint_as_float(x); }

// Packed fp32 pairs: the f32x2 forms of add and fma do the work of two scalar instructions in one
// issue slot, each half rounded exactly as the scalar instruction rounds it.
__device__ __forceinline__ uint64_t pk2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ float2 up2(uint64_t x) {
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(x));
    return r;
}
__device__ __forceinline__ uint64_t fma2(uint64_t x, uint64_t y, uint64_t z) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(x), "l"(y), "l"(z));
    return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t x, uint64_t y) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(x), "l"(y));
    return d;
}
__device__ __forceinline__ uint64_t ex2_2(uint64_t x) {     // 2^x of both halves, on the SFU
    const float2 t = up2(x);
    return pk2(ex2(t.x), ex2(t.y));
}
// 2^(S*a + z) for the element pair (v[c], v[c+1])
__device__ __forceinline__ uint64_t p2(const uint32_t (&v)[16], int c, uint64_t a2, uint64_t z2) {
    return ex2_2(fma2(pk2(f(v[c]), f(v[c + 1])), a2, z2));
}

// pass 1, one 16-column chunk of one query row, every column visible: online (m, l) in base 2,
// m = max S*a, l = sum 2^(S*a - m); the running sum is rescaled only when the max grows
__device__ __forceinline__ void row_chunk_full(const uint32_t (&v)[16], float a, float& m, float& l) {
    const float x0 = max3(f(v[0]), f(v[1]), f(v[2])), x1 = max3(f(v[3]), f(v[4]), f(v[5]));
    const float x2 = max3(f(v[6]), f(v[7]), f(v[8])), x3 = max3(f(v[9]), f(v[10]), f(v[11]));
    const float x4 = max3(f(v[12]), f(v[13]), f(v[14]));
    const float mx = max3(max3(x0, x1, x2), max3(x3, x4, f(v[15])), x0) * a;
    if (mx > m) {
        l *= ex2(m - mx);
        m = mx;
    }
    const uint64_t a2 = pk2(a, a), nm2 = pk2(-m, -m);
    uint64_t s0 = p2(v, 0, a2, nm2), s1 = p2(v, 2, a2, nm2);
#pragma unroll
    for (int c = 4; c < 16; c += 4) {
        s0 = add2(s0, p2(v, c, a2, nm2));
        s1 = add2(s1, p2(v, c + 2, a2, nm2));
    }
    const float2 t = up2(add2(s0, s1));
    l += t.x + t.y;
}

// pass 1 with the causal limit: columns c <= lim are visible
__device__ __forceinline__ void row_chunk_masked(const uint32_t (&v)[16], int lim, float a, float& m, float& l) {
    if (lim < 0) return;
    float mx = -INFINITY;
#pragma unroll
    for (int c = 0; c < 16; ++c)
        if (c <= lim) mx = fmaxf(mx, f(v[c]));
    mx *= a;
    if (mx > m) {
        l *= ex2(m - mx);
        m = mx;
    }
    float sm = 0.f;
#pragma unroll
    for (int c = 0; c < 16; ++c)
        if (c <= lim) sm += ex2(fmaf(f(v[c]), a, -m));
    l += sm;
}

// pass 2, one 16-column chunk of one key, every row visible: sum of 2^(S*a - c_row); ncv holds -c_row
// (-inf for rows that are not window rows of this request, which therefore contribute 0).  The sum
// is kept as two packed pairs.
__device__ __forceinline__ void key_chunk_full(const uint32_t (&v)[16], const float* ncv, float a, uint64_t (&acc)[2]) {
    const float4* nc4 = reinterpret_cast<const float4*>(ncv);
    const uint64_t a2 = pk2(a, a);
#pragma unroll
    for (int c = 0; c < 16; c += 4) {
        const float4 n = nc4[c / 4];
        acc[0] = add2(acc[0], p2(v, c, a2, pk2(n.x, n.y)));
        acc[1] = add2(acc[1], p2(v, c + 2, a2, pk2(n.z, n.w)));
    }
}

// pass 2 for slices of eight chunks (one whole job per warpgroup): the chunk's normalisers come from
// the lanes that hold them by warp shuffle instead of broadcast shared-memory loads, which compete with
// the MMA's shared-memory operand reads.  Lane L holds -c of column 32 * r + L of the slice in cr
// (r = chunk / 2); the chunk's column 16 * half + i of that 32-column group comes from lane 16 * half + i.
__device__ __forceinline__ void key_chunk_full_sh(const uint32_t (&v)[16], float cr, int half, float a,
                                                  uint64_t (&acc)[2]) {
    const uint64_t a2 = pk2(a, a);
#pragma unroll
    for (int c = 0; c < 16; c += 4) {
        const float n0 = __shfl_sync(0xffffffffu, cr, half * 16 + c);
        const float n1 = __shfl_sync(0xffffffffu, cr, half * 16 + c + 1);
        const float n2 = __shfl_sync(0xffffffffu, cr, half * 16 + c + 2);
        const float n3 = __shfl_sync(0xffffffffu, cr, half * 16 + c + 3);
        acc[0] = add2(acc[0], p2(v, c, a2, pk2(n0, n1)));
        acc[1] = add2(acc[1], p2(v, c + 2, a2, pk2(n2, n3)));
    }
}

// pass 2 with the causal mask: key i is visible to the query row at local position pos iff i <= pos.
// The slab's rows are head-major (row qg is window position qg % n of head qg / n) and qg0 and n are
// multiples of 16, so the chunk's 16 rows are window positions t0 .. t0 + 15 of one head: one modulo
// per chunk instead of one per element.
__device__ __forceinline__ void key_chunk_masked(const uint32_t (&v)[16], const float* ncv, float a, int i, int qg0,
                                                 int n, int N, int rows_total, uint64_t (&acc)[2]) {
    if (i >= N) return;
    const int t0 = qg0 % n;
    const int lim = i - (N - n + t0);              // column c is visible iff c >= lim (pos = N - n + t0 + c >= i)
    const int rows_left = rows_total - qg0;        // and c < rows_left
    float s[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int c = 0; c < 16; ++c) {
        const bool vis = c >= lim && c < rows_left && N - n + t0 + c >= 0;
        const float p = ex2(fmaf(f(v[c]), a, ncv[c]));
        s[c & 3] += vis ? p : 0.f;
    }
    acc[0] = add2(acc[0], pk2(s[0], s[1]));
    acc[1] = add2(acc[1], pk2(s[2], s[3]));
}

__device__ __forceinline__ void release_tmem(const Smem& S, uint32_t buf, int lane) {
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(S.tempty + buf));
}

// One job slice whose every element is visible to every thread of the warp: NCH 16-column chunks,
// TMEM loads double-buffered (the next chunk in flight while the current one is reduced); the TMEM
// buffer is released as soon as its last chunk has landed.  Straight-line code, kept compact.
// Pass 1 updates (m, l) of this thread's row; pass 2 adds into this thread's key sum.
template <int PASS, int NCH>
__device__ __forceinline__ void run_job_fast(const Smem& S, uint32_t ta, uint32_t buf, int lane, float a,
                                             const float* ncv0, float& m, float& l, uint64_t (&acc)[2]) {
    constexpr bool kShfl = PASS == 2 && NCH == 8;
    uint32_t va[16], vb[16];
    float creg[NCH / 2];
    if (kShfl) {
#pragma unroll
        for (int r = 0; r < NCH / 2; ++r) creg[r] = ncv0[32 * r + lane];
    }
    tmem_ld16(ta, va);
    tmem_wait_pin(va);
#pragma unroll
    for (int ch = 0; ch < NCH; ch += 2) {
        tmem_ld16(ta + (ch + 1) * 16, vb);
        if (PASS == 1) row_chunk_full(va, a, m, l);
        else if (kShfl) key_chunk_full_sh(va, creg[ch / 2], 0, a, acc);
        else key_chunk_full(va, ncv0 + ch * 16, a, acc);
        tmem_wait_pin(vb);
        if (ch + 2 < NCH) tmem_ld16(ta + (ch + 2) * 16, va);
        else release_tmem(S, buf, lane);
        if (PASS == 1) row_chunk_full(vb, a, m, l);
        else if (kShfl) key_chunk_full_sh(vb, creg[ch / 2], 1, a, acc);
        else key_chunk_full(vb, ncv0 + (ch + 1) * 16, a, acc);
        if (ch + 2 < NCH) tmem_wait_pin(va);
    }
}

// The general case (tiles that reach into the causal window or past the request's end, and the
// abort path, which reads nothing and only releases the buffer): one chunk at a time with the masks.
// Pass 1: columns up to lim0 (relative to the slice's first column) of a valid row; pass 2: key
// `key` against the slice's rows qg0.. of a request of N tokens.
template <int PASS>
__device__ __forceinline__ void run_job_slow(const Smem& S, uint32_t ta, uint32_t buf, int lane, bool ok, int nch,
                                             float a, bool rvalid, int lim0, const float* ncv0, int key, int qg0,
                                             int n, int N, int rows_total, float& m, float& l, uint64_t (&acc)[2]) {
    for (int ch = 0; ch < nch; ++ch) {
        uint32_t v[16];
        if (ok) {
            tmem_ld16(ta + ch * 16, v);
            tmem_wait_pin(v);
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = 0u;
        }
        if (ch == nch - 1) release_tmem(S, buf, lane);
        if (!ok) continue;
        if (PASS == 1) {
            if (rvalid) row_chunk_masked(v, lim0 - ch * 16, a, m, l);
        } else {
            key_chunk_masked(v, ncv0 + ch * 16, a, key, qg0 + ch * 16, n, N, rows_total, acc);
        }
    }
}

template <int PASS, int NCH>
__device__ void epilogue(const Params& P, const Smem& S, uint32_t tmem_base, int it0, int it1) {
    if (PASS == 2) pdl_wait();                  // the normalisers (merge kernel) are read below
    volatile int* abort_flag = S.abort_flag;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int et = threadIdx.x - 64;            // 0..511
    const int wg = (warp - 2) >> 2;             // warpgroup 0..3
    const int q = warp & 3;                     // TMEM lane quarter this warp may access
    const int rl = q * 32 + lane;               // row (pass 1) or key (pass 2) inside a 128-tile
    const float a = P.a;
    const JobMap jm = job_map<PASS>(P);
    const int J = jm.J;
    const int wpj = jm.wpj;                     // warpgroups per job
    const int cols = NCH * 16;                  // columns this warpgroup reads per job = W / wpj
    const int col0 = (wpj == 1 ? 0 : (wg % wpj) * cols);
    const int jfirst = wg / wpj;
    const int jstep = 4 / wpj;
    const uint32_t tl = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + col0;
    uint32_t tiles_done = 0;
    int prev_unit = -1, prev_slab = -1;
    uint32_t tile_par = 0;
    float m0 = -INFINITY, l0 = 0.f, m1 = -INFINITY, l1 = 0.f;   // pass 1 state of the (<= 2) jobs
    // pass 1: this thread's row in each of its (<= 2) jobs: inside the slab's rows, and its position
    // in the window (qg % n); set when the slab changes
    bool rin0 = false, rin1 = false;
    int rmod0 = 0, rmod1 = 0;

    for (int it = it0; it < it1; ++it) {
        int4 ia, ib;
        item_load(P, it, it1, ia, ib);
        const ItemInfo I = item_decode(P, ia, ib);
        const int ne = min(P.n, I.N);
        const int row0 = I.slab * P.slab_rows;   // first global query row of this slab
        if (PASS == 2 && I.unit != prev_unit) {
            named_bar_sync(1, kEpiThreads);
            for (int i = et; i < P.slab_rows; i += kEpiThreads)
                S.cvec[i] = UP_IN((int64_t)I.unit * P.slab_rows + i, P.lim_cvec, P.status)
                                ? -__ldcg(P.cvec + (size_t)I.unit * P.slab_rows + i) : -INFINITY;
            named_bar_sync(1, kEpiThreads);
        }
        prev_unit = I.unit;
        if (PASS == 1 && I.slab != prev_slab) {
            const int q0 = row0 + jfirst * 128 + rl, q1 = q0 + jstep * 128;
            rin0 = jfirst < J && q0 < P.rows_total;
            rin1 = jfirst + jstep < J && q1 < P.rows_total;
            rmod0 = q0 % P.n;
            rmod1 = q1 % P.n;
            prev_slab = I.slab;
        }
        if (PASS == 1) {
            m0 = m1 = -INFINITY;
            l0 = l1 = 0.f;
        }
        for (int kt = I.tb; kt < I.te; ++kt, ++tiles_done) {
            uint64_t acc[2] = {0ull, 0ull};                 // pass 2: packed (+0.0f, +0.0f) pairs
            const bool tile_full = kt * kTileKeys + kTileKeys - 1 <= I.N - ne;
            int u = 0;
            for (int j = jfirst; j < J; j += jstep, ++u) {
                const uint32_t jc = tiles_done * J + j;
                const uint32_t buf = jc & (jm.nbuf - 1);
                const bool ok =
                    __all_sync(0xffffffffu, mbar_wait(smem_u32(S.tfull + buf), (jc >> jm.nb_log) & 1, abort_flag));
                tc_fence_after();
                const uint32_t ta = tl + buf * jm.W;
                const float* ncv0 = S.cvec + j * jm.W + col0;
                float mm = u ? m1 : m0, ll = u ? l1 : l0;
                bool rvalid = false;
                int lim0 = 0;
                bool fast;
                if (PASS == 1) {
                    const int pos = I.N - P.n + (u ? rmod1 : rmod0);    // this thread's row position
                    rvalid = (u ? rin1 : rin0) && pos >= 0;
                    lim0 = pos - (kt * kTileKeys + col0);               // last visible column of the slice
                    fast = rvalid && lim0 >= cols - 1;
                } else {
                    fast = tile_full;
                }
                if (ok && __all_sync(0xffffffffu, fast))
                    run_job_fast<PASS, NCH>(S, ta, buf, lane, a, ncv0, mm, ll, acc);
                else
                    run_job_slow<PASS>(S, ta, buf, lane, ok, NCH, a, rvalid, lim0, ncv0, kt * kTileKeys + rl,
                                       row0 + j * jm.W + col0, P.n, I.N, P.rows_total, mm, ll, acc);
                if (PASS == 1) {
                    if (u) { m1 = mm; l1 = ll; } else { m0 = mm; l0 = ll; }
                }
            }
            if (PASS == 2) {
                // this warpgroup's per-key partial, reduced over G consecutive keys (keys are TMEM lanes,
                // so warp shuffles, then the warps of the group for G > 32); one partial per warpgroup
                const float2 t01 = up2(acc[0]), t23 = up2(acc[1]);
                const float tot = (t01.x + t01.y) + (t23.x + t23.y);
                const int i = kt * kTileKeys + rl;
                const size_t part = (size_t)I.kk * 4 + wg;
                if (P.tok != nullptr && i < I.N && UP_IN(part * P.T + I.base + i, P.lim_tok, P.status))
                    P.tok[part * P.T + I.base + i] = tot;
                const int nb = (I.N + P.G - 1) / P.G;
                float* dst = P.blk + part * P.nb_cap + P.cb[I.r];
                float s = tot;
                const int gw = P.G < 32 ? P.G : 32;
                for (int o = gw >> 1; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
                if (P.G <= 32) {
                    const int g = i / P.G;
                    if ((lane & (P.G - 1)) == 0 && g < nb && UP_IN(dst + g - P.blk, P.lim_blk, P.status)) dst[g] = s;
                } else {
                    float* wsum = reinterpret_cast<float*>(S.xchg) + (tile_par & 1) * 16 + wg * 4;
                    if (lane == 0) wsum[q] = s;
                    named_bar_sync(2 + wg, 128);
                    if (lane == 0) {
                        if (P.G == 64 && (q & 1) == 0) {
                            const int g = i / 64;
                            if (g < nb && UP_IN(dst + g - P.blk, P.lim_blk, P.status)) dst[g] = wsum[q] + wsum[q + 1];
                        } else if (P.G == 128 && q == 0) {
                            const int g = i / 128;
                            if (g < nb && UP_IN(dst + g - P.blk, P.lim_blk, P.status))
                                dst[g] = (wsum[0] + wsum[1]) + (wsum[2] + wsum[3]);
                        }
                    }
                }
                ++tile_par;
            }
        }
        if (PASS == 1) {
            // merge the warpgroups that share a job (fixed order), write this item's partial (m, l)
            // into the unit's block, laid out [row][item of the unit] for the merge kernel
            const int2 ui = I.ui;
            float2* part = P.ml + (size_t)ui.x * P.slab_rows + I.tb / kItemTiles;   // tile pair in the unit
            float2* xm = reinterpret_cast<float2*>(S.xchg);             // [4 warpgroups][2 jobs][128 rows]
            if (wpj > 1) {
                int u = 0;
                for (int j = jfirst; j < J; j += jstep, ++u)
                    xm[(wg * 2 + u) * 128 + rl] = u ? make_float2(m1, l1) : make_float2(m0, l0);
                named_bar_sync(1, kEpiThreads);
                if (wg % wpj == 0) {
                    u = 0;
                    for (int j = jfirst; j < J; j += jstep, ++u) {
                        float mm = -INFINITY;
                        for (int w2 = wg; w2 < wg + wpj; ++w2) mm = fmaxf(mm, xm[(w2 * 2 + u) * 128 + rl].x);
                        float ll = 0.f;
                        if (mm > -INFINITY)
                            for (int w2 = wg; w2 < wg + wpj; ++w2) {
                                const float2 e = xm[(w2 * 2 + u) * 128 + rl];
                                ll += e.y * ex2(e.x - mm);
                            }
                        if (UP_IN(part + (size_t)(j * 128 + rl) * ui.y - P.ml, P.lim_ml, P.status))
                            part[(size_t)(j * 128 + rl) * ui.y] = make_float2(mm, ll);
                    }
                }
                named_bar_sync(1, kEpiThreads);
            } else {
                int u = 0;
                for (int j = jfirst; j < J; j += jstep, ++u)
                    if (UP_IN(part + (size_t)(j * 128 + rl) * ui.y - P.ml, P.lim_ml, P.status))
                        part[(size_t)(j * 128 + rl) * ui.y] = u ? make_float2(m1, l1) : make_float2(m0, l0);
            }
        }
    }
}

// ------------------------------------------------------------------------------------------------
// the one pass: row statistics and block sums from a single Q.K^T
//
// Per window row j and key tile t, with a running maximum m_t (base 2, over the keys seen up to the end
// of tile t) the epilogue computes the sums
//   e_{j,g} = sum_{i in B_g} 2^(S_ji * a - m_t)      for the 128 / G blocks g of tile t
// and writes them with m_t (at d_k = 256 the two threads that read the halves of row j's tile each sum
// against their own maximum and rescale to the larger one before writing).  The (m, l) partials per
// work item (merged over the threads that hold a row) are written as in pass 1, so the merge kernel
// gives c_j = m_j + log2(l_j), and the reduce kernel then forms Eq. 4 exactly:
//   sum_j sum_{i in B_g} A_ji = sum_j e_{j,g} * 2^(m_t - c_j).
// This is the two-pass softmax of the section 3.5 kernel design with the second pass run over the block
// sums (G times smaller than S) instead of over a recomputed S: the tensor work and the exponentials of
// the recompute pass disappear; S itself is never stored.

// columns 16*ch + c > lim of a chunk become -inf (keys after the row's position, or a row that is not a
// window row of this request: lim < 0)
__device__ __forceinline__ void mask_chunk(uint32_t (&v)[16], int ch, int lim) {
#pragma unroll
    for (int c = 0; c < 16; ++c)
        if (16 * ch + c > lim) v[c] = 0xFF800000u;
}

// 32 columns (the 16-column chunks 2*h2 and 2*h2+1 of this thread's half-tile) of its row in the one
// pass: fold their maximum into m (rescaling the sub-block sums of the half-tile so far and the l of the
// item's earlier tiles when it grows), then add 2^(S*a - m) over each chunk to its sub-block's sum
// e[chunk / CPB] (CPB = G / 16 chunks per block; a 128-key block has one sub-block per half).  One
// maximum update per 32 columns leaves 32 independent exponentials behind it (measured 2-8% faster
// score calls than an update per 16 columns).  Columns outside the causal range arrive as -inf and add 0.
template <int CPB, int NE>
__device__ __forceinline__ void one_pass_chunk32(const uint32_t (&v)[32], int h2, float a, float& m, float& l,
                                                 float (&e)[NE]) {
    float x[6];
#pragma unroll
    for (int i = 0; i < 5; ++i) x[i] = max3(f(v[6 * i]), f(v[6 * i + 1]), f(v[6 * i + 2]));
    x[5] = max3(f(v[3]), f(v[4]), f(v[5]));
    float y0 = max3(f(v[9]), f(v[10]), f(v[11])), y1 = max3(f(v[15]), f(v[16]), f(v[17]));
    float y2 = max3(f(v[21]), f(v[22]), f(v[23])), y3 = max3(f(v[27]), f(v[28]), f(v[29]));
    const float z = max3(f(v[30]), f(v[31]), x[0]);
    const float mx = max3(max3(x[1], x[2], x[3]), max3(x[4], x[5], z), max3(y0, y1, max(y2, y3))) * a;
    if (mx > m) {
        const float sc = ex2(m - mx);           // 0 while m = -inf
        l *= sc;
#pragma unroll
        for (int b = 0; b < NE; ++b)
            if (b <= (2 * h2 + 1) / CPB) e[b] *= sc;
        m = mx;
    }
    // while m is -inf every value so far is -inf: any finite reference gives the sum 0, not NaN
    const float mr = m == -INFINITY ? 0.f : m;
    const uint64_t a2 = pk2(a, a), nm2 = pk2(-mr, -mr);
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
        const uint32_t(&w)[16] = *reinterpret_cast<const uint32_t(*)[16]>(&v[16 * hf]);
        uint64_t s0 = p2(w, 0, a2, nm2), s1 = p2(w, 2, a2, nm2);
#pragma unroll
        for (int c = 4; c < 16; c += 4) {
            s0 = add2(s0, p2(w, c, a2, nm2));
            s1 = add2(s1, p2(w, c + 2, a2, nm2));
        }
        const float2 t = up2(add2(s0, s1));
        e[(2 * h2 + hf) / CPB] += t.x + t.y;
    }
}

// one half-tile (64 columns) of one job for this thread's row, the TMEM buffer released as soon as its
// last columns have landed; `masked` (warp-uniform) applies the causal limit lim (relative to the
// half's first column)
template <int CPB, int NE>
__device__ __forceinline__ void one_pass_half(const Smem& S, uint32_t ta, uint32_t buf, int lane, bool masked, int lim,
                                              float a, float& m, float& l, float (&e)[NE]) {
    // two 32-column loads, the second in flight while the first is reduced
    uint32_t va[32], vb[32];
    tmem_ld32(ta, va);
    tmem_wait_pin32(va);
    tmem_ld32(ta + 32, vb);
    if (masked) {
        mask_chunk(*reinterpret_cast<uint32_t(*)[16]>(&va[0]), 0, lim);
        mask_chunk(*reinterpret_cast<uint32_t(*)[16]>(&va[16]), 1, lim);
    }
    one_pass_chunk32<CPB, NE>(va, 0, a, m, l, e);
    tmem_wait_pin32(vb);
    release_tmem(S, buf, lane);
    if (masked) {
        mask_chunk(*reinterpret_cast<uint32_t(*)[16]>(&vb[0]), 2, lim);
        mask_chunk(*reinterpret_cast<uint32_t(*)[16]>(&vb[16]), 3, lim);
    }
    one_pass_chunk32<CPB, NE>(vb, 1, a, m, l, e);
}

// one whole 128-column job of this thread's row, the buffer released as soon as its last columns have
// landed; `masked` (warp-uniform) applies the causal limit lim
template <int CPB>
__device__ __forceinline__ void one_pass_tile(const Smem& S, uint32_t ta, uint32_t buf, int lane, bool masked, int lim,
                                              float a, float& m, float& l, float (&e)[8 / CPB]) {
    // 32-column loads, double-buffered: the load of the next 32 columns is in flight while the current
    // 32 are reduced with one maximum update
    uint32_t va[32], vb[32];
    tmem_ld32(ta, va);
    tmem_wait_pin32(va);
#pragma unroll
    for (int h = 0; h < 4; h += 2) {
        tmem_ld32(ta + (h + 1) * 32, vb);
        if (masked) {
            mask_chunk(*reinterpret_cast<uint32_t(*)[16]>(&va[0]), 2 * h, lim);
            mask_chunk(*reinterpret_cast<uint32_t(*)[16]>(&va[16]), 2 * h + 1, lim);
        }
        one_pass_chunk32<CPB, 8 / CPB>(va, h, a, m, l, e);
        tmem_wait_pin32(vb);
        if (h + 2 < 4) tmem_ld32(ta + (h + 2) * 32, va);
        else release_tmem(S, buf, lane);
        if (masked) {
            mask_chunk(*reinterpret_cast<uint32_t(*)[16]>(&vb[0]), 2 * h + 2, lim);
            mask_chunk(*reinterpret_cast<uint32_t(*)[16]>(&vb[16]), 2 * h + 3, lim);
        }
        one_pass_chunk32<CPB, 8 / CPB>(vb, h + 1, a, m, l, e);
        if (h + 2 < 4) tmem_wait_pin32(va);
    }
}

// d_k <= 128 (the jobs-outer issue order): warpgroup w drains TMEM buffer w whole; with J in {1, 2, 4}
// jobs per tile that is always job w % J (the same 128 window rows), on every (4 / J)-th tile of the
// CTA's sequence.  (The pairs of epilogue_one_pass_pairs measured 20-35% slower here: a thread then
// pays the first TMEM load and the per-job bookkeeping twice per tile.)  The warpgroups that hold the
// same rows merge their (m, l) at the end of each item in a fixed order, as in pass 1.  CPB = G / 16.
template <int CPB>
__device__ void epilogue_one_pass_whole(const Params& P, const Smem& S, uint32_t tmem_base, int it0, int it1) {
    constexpr int SPT = 8 / CPB;                // blocks per tile
    volatile int* abort_flag = S.abort_flag;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int wg = (warp - 2) >> 2;             // warpgroup 0..3 = the TMEM buffer it drains
    const int q = warp & 3;                     // TMEM lane quarter this warp may access
    const int rl = q * 32 + lane;
    const int J = P.J;
    const int j = wg % J;                       // the job (128 rows of the slab) of this warpgroup
    const int row = j * 128 + rl;               // this thread's row in the slab
    const float a = P.a;
    const uint32_t ta = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + wg * 128;
    uint32_t tiles_done = 0;
    int prev_slab = -1;
    bool rin = false;
    int rmod = 0;
    for (int it = it0; it < it1; ++it) {
        int4 ia, ib;
        item_load(P, it, it1, ia, ib);
        const ItemInfo I = item_decode(P, ia, ib);
        if (I.slab != prev_slab) {
            const int qg = I.slab * P.slab_rows + row;
            rin = qg < P.rows_total;
            rmod = qg % P.n;
            prev_slab = I.slab;
        }
        const int pos = I.N - P.n + rmod;       // this row's position in the request
        const bool rvalid = rin && pos >= 0;
        const int2 ui = I.ui;
        const size_t tile0 = static_cast<size_t>(ui.x) * kItemTiles;   // the unit's first key tile
        float m = -INFINITY, l = 0.f;
        for (int kt = I.tb; kt < I.te; ++kt, ++tiles_done) {
            const uint32_t jc = tiles_done * J + j;
            if ((jc & 3u) != static_cast<uint32_t>(wg)) continue;           // another warpgroup's tile
            const bool ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(S.tfull + wg), (jc >> 2) & 1, abort_flag));
            tc_fence_after();
            if (!ok) {
                release_tmem(S, wg, lane);
                continue;
            }
            const int lim = rvalid ? pos - kt * kTileKeys : -1;               // last visible column
            float e[SPT];
#pragma unroll
            for (int b = 0; b < SPT; ++b) e[b] = 0.f;
            const bool masked = !__all_sync(0xffffffffu, lim >= kTileKeys - 1);
            one_pass_tile<CPB>(S, ta, wg, lane, masked, lim, a, m, l, e);
            const size_t t = tile0 + kt;
            if (UP_IN(t * P.slab_rows + row, P.lim_bm, P.status)) P.bm[t * P.slab_rows + row] = m;
            float* dst = P.be + t * SPT * P.slab_rows + row;
            float ts = 0.f;
#pragma unroll
            for (int b = 0; b < SPT; ++b) {
                if (UP_IN(dst + static_cast<size_t>(b) * P.slab_rows - P.be, P.lim_be, P.status))
                    dst[static_cast<size_t>(b) * P.slab_rows] = e[b];
                ts += e[b];
            }
            l += ts;
        }
        // this item's (m, l) partial of the row, merged over the 4 / J warpgroups that hold the row
        float2* part = P.ml + (size_t)ui.x * P.slab_rows + I.tb / kItemTiles;
        if (J == 4) {
            if (UP_IN(part + (size_t)row * ui.y - P.ml, P.lim_ml, P.status)) part[(size_t)row * ui.y] = make_float2(m, l);
        } else {
            float2* xm = reinterpret_cast<float2*>(S.xchg);                  // [4 warpgroups][128 rows]
            xm[wg * 128 + rl] = make_float2(m, l);
            named_bar_sync(1, kEpiThreads);
            if (wg < J) {
                float mm = -INFINITY;
                for (int w2 = wg; w2 < 4; w2 += J) mm = fmaxf(mm, xm[w2 * 128 + rl].x);
                float ll = 0.f;
                if (mm > -INFINITY)
                    for (int w2 = wg; w2 < 4; w2 += J) {
                        const float2 x = xm[w2 * 128 + rl];
                        ll += x.y * ex2(x.x - mm);
                    }
                if (UP_IN(part + (size_t)row * ui.y - P.ml, P.lim_ml, P.status)) part[(size_t)row * ui.y] = make_float2(mm, ll);
            }
            named_bar_sync(1, kEpiThreads);
        }
    }
}

// d_k = 256 (the chunks-outer issue order, J = 1 or 2 jobs per tile): the four epilogue warpgroups
// form two pairs; pair p drains the jobs q (running job count) with q mod 2 = p, which are those in
// TMEM buffers p and p + 2, and in each job warpgroup 2p + h reads the columns 64h .. 64h + 63.  With
// J = 2 a pair holds the rows of job p; with J = 1 the pairs take alternate tiles of the one job.  A
// job is drained by eight warps, so its TMEM buffer comes free in about half the time one warpgroup
// takes, and consecutive jobs drain on different pairs.  Each half keeps its own running maximum; at
// the end of a job the two threads of a row trade (maximum, sum) through shared memory and write the
// tile's block sums against the larger maximum, so the output is the same (m_t, e_{j,g}) as with one
// thread per row.  The threads that hold a row merge their (m, l) at the end of each item in a fixed
// order, as in pass 1.  CPB = G / 16.
template <int CPB>
__device__ void epilogue_one_pass_pairs(const Params& P, const Smem& S, uint32_t tmem_base, int it0, int it1) {
    constexpr int NE = sub_blocks_per_half(16 * CPB);   // sums per half-tile: its blocks, or half of one
    constexpr int SPT = 8 / CPB;                         // blocks per tile
    volatile int* abort_flag = S.abort_flag;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int wg = (warp - 2) >> 2;             // warpgroup 0..3
    const int pair = wg >> 1, h = wg & 1;       // jobs q with q % 2 == pair; columns 64h ..
    const int qd = warp & 3;                    // TMEM lane quarter this warp may access
    const int rl = qd * 32 + lane;
    const int J = P.J;                          // 1 or 2
    const int job = J == 2 ? pair : 0;          // the job (128 rows of the slab) of this thread's row
    const int row = job * 128 + rl;
    const float a = P.a;
    const uint32_t ta0 = tmem_base + (static_cast<uint32_t>(qd * 32) << 16) + 64 * h;
    uint32_t tiles_done = 0, jn = 0;
    int prev_slab = -1;
    bool rin = false;
    int rmod = 0;
    for (int it = it0; it < it1; ++it) {
        int4 ia, ib;
        item_load(P, it, it1, ia, ib);
        const ItemInfo I = item_decode(P, ia, ib);
        if (I.slab != prev_slab) {
            const int qg = I.slab * P.slab_rows + row;
            rin = qg < P.rows_total;
            rmod = qg % P.n;
            prev_slab = I.slab;
        }
        const int pos = I.N - P.n + rmod;       // this row's position in the request
        const bool rvalid = rin && pos >= 0;
        const int2 ui = I.ui;
        const size_t tile0 = static_cast<size_t>(ui.x) * kItemTiles;   // the unit's first key tile
        float m = -INFINITY, l = 0.f;
        for (int kt = I.tb; kt < I.te; ++kt, ++tiles_done) {
            const uint32_t q = tiles_done * J + job;
            if ((q & 1u) != static_cast<uint32_t>(pair)) continue;          // the other pair's tile (J = 1)
            const uint32_t buf = q & 3u;
            const bool ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(S.tfull + buf), (q >> 2) & 1, abort_flag));
            tc_fence_after();
            float e[NE];
#pragma unroll
            for (int b = 0; b < NE; ++b) e[b] = 0.f;
            if (ok) {
                const int lim = rvalid ? pos - kt * kTileKeys - 64 * h : -1;      // last visible column
                const bool masked = !__all_sync(0xffffffffu, lim >= 63);
                one_pass_half<CPB, NE>(S, ta0 + buf * 128, buf, lane, masked, lim, a, m, l, e);
            } else {
                release_tmem(S, buf, lane);
            }
            // the other half's (maximum, sum): double-buffered by job so that one pair barrier per job
            // suffices (a half writes job k + 2's entry only after both passed job k + 1's barrier);
            // every thread of the pair reaches it, whatever `ok` was
            float2* xj = reinterpret_cast<float2*>(S.cvec) + ((jn & 1u) * 2 + pair) * 256;   // [half][128]
            xj[h * 128 + rl] = make_float2(m, e[0]);
            named_bar_sync(1 + pair, kEpiThreads / 2);
            const float2 o = xj[(h ^ 1) * 128 + rl];
            ++jn;
            const float M = fmaxf(m, o.x);
            const float sc = m == -INFINITY ? 0.f : ex2(m - M);               // this half's sums to M
            const size_t t = tile0 + kt;
            float ts = 0.f;
#pragma unroll
            for (int b = 0; b < NE; ++b) ts += e[b];
            l += ts;
            if (!ok) continue;
            if (SPT == 1) {
                // G = 128: the tile's one block spans both halves
                if (h == 0) {
                    const float so = o.x == -INFINITY ? 0.f : ex2(o.x - M);
                    if (UP_IN(t * P.slab_rows + row, P.lim_be, P.status)) P.be[t * P.slab_rows + row] = e[0] * sc + o.y * so;
                }
            } else {
#pragma unroll
                for (int b = 0; b < NE; ++b) {
                    const size_t ei = (t * SPT + h * NE + b) * P.slab_rows + row;
                    if (UP_IN(ei, P.lim_be, P.status)) P.be[ei] = e[b] * sc;
                }
            }
            if (h == 0 && UP_IN(t * P.slab_rows + row, P.lim_bm, P.status)) P.bm[t * P.slab_rows + row] = M;
        }
        // this item's (m, l) partial of the row, merged over the threads that hold it: the two halves of
        // its pair (a barrier of the pair only, so that the pairs stay independent), and with J = 1 both
        // pairs
        float2* part = P.ml + (size_t)ui.x * P.slab_rows + I.tb / kItemTiles;
        float2* xm = reinterpret_cast<float2*>(S.xchg);                      // [4 warpgroups][128]
        xm[wg * 128 + rl] = make_float2(m, l);
        const int bar_id = J == 2 ? 1 + pair : 3, bar_n = J == 2 ? kEpiThreads / 2 : kEpiThreads;
        named_bar_sync(bar_id, bar_n);
        const int wfirst = J == 2 ? 2 * pair : 0, wcount = J == 2 ? 2 : 4;
        if (wg == wfirst) {
            float mm = -INFINITY;
            for (int w2 = wfirst; w2 < wfirst + wcount; ++w2) mm = fmaxf(mm, xm[w2 * 128 + rl].x);
            float ll = 0.f;
            if (mm > -INFINITY)
                for (int w2 = wfirst; w2 < wfirst + wcount; ++w2) {
                    const float2 x = xm[w2 * 128 + rl];
                    ll += x.y * ex2(x.x - mm);
                }
            if (UP_IN(part + (size_t)row * ui.y - P.ml, P.lim_ml, P.status)) part[(size_t)row * ui.y] = make_float2(mm, ll);
        }
        named_bar_sync(bar_id, bar_n);
    }
}

// Fold each query row's pass-1 partials (one per work item of its unit, in the unit's key-tile order)
// into c = m + log2(l): one warp per (unit, row), lanes over the items, fixed shuffle trees.
// warp gw of nw (whole warps) folds the rows gw, gw + nw, ...
__device__ void merge_rows(const Params& P, int64_t gw, int64_t nw) {
    const int lane = threadIdx.x & 31;
    const int64_t rows_all = (int64_t)P.R * P.units_per_req * P.slab_rows;
    for (int64_t gr = gw; gr < rows_all; gr += nw) {
        const int u = static_cast<int>(gr / P.slab_rows), row = static_cast<int>(gr % P.slab_rows);
        const int2 ui = __ldcg(&P.unit_items[u]);
        const float2* part = P.ml + (size_t)ui.x * P.slab_rows + (size_t)row * ui.y;
        if (!UP_IN(u, P.lim_units, P.status) || !UP_IN(part + ui.y - 1 - P.ml, P.lim_ml, P.status)) continue;
        // the first kCache partials of each lane stay in registers between the max and the sum (one
        // round of loads instead of two); the sum keeps its order (p = lane, lane + 32, ...)
        constexpr int kCache = 8;
        float2 e[kCache];
        float mm = -INFINITY;
#pragma unroll
        for (int i = 0; i < kCache; ++i) {
            const int p = lane + 32 * i;
            e[i] = p < ui.y ? __ldcg(&part[p]) : make_float2(-INFINITY, 0.f);
            mm = fmaxf(mm, e[i].x);
        }
        for (int p = lane + 32 * kCache; p < ui.y; p += 32) mm = fmaxf(mm, __ldcg(&part[p].x));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mm = fmaxf(mm, __shfl_xor_sync(0xffffffffu, mm, o));
        float ll = 0.f;
        if (mm > -INFINITY) {
#pragma unroll
            for (int i = 0; i < kCache; ++i)
                if (e[i].x > -INFINITY) ll += e[i].y * ex2(e[i].x - mm);     // an empty partial adds 0
            for (int p = lane + 32 * kCache; p < ui.y; p += 32) {
                const float2 x = __ldcg(&part[p]);
                ll += x.y * ex2(x.x - mm);
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ll += __shfl_xor_sync(0xffffffffu, ll, o);
        if (lane == 0 && UP_IN((size_t)u * P.slab_rows + row, P.lim_cvec, P.status))
            P.cvec[(size_t)u * P.slab_rows + row] = mm == -INFINITY ? INFINITY : mm + log2f(ll);
    }
}

__global__ void __launch_bounds__(256) merge_kernel(Params P) {
    pdl_wait();
    pdl_trigger();
    if (__ldcg(P.n_items + 1) == 0) return;
    merge_rows(P, (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5), (int64_t)gridDim.x * (blockDim.x >> 5));
}

// The one pass's Eq. 4: a CTA forms the SPT = 128 / G block scores of one (request, key tile) at a time
//   b_g = 1/(n_eff * Hq * G) * sum over the request's units and their rows j of e_{j,g} * 2^(m_t,j - c_j)
// (each CTA takes a contiguous range of these tasks).  Threads take (unit, group of 4 rows) pairs in a
// fixed assignment, with 16-byte loads, several pairs' loads in flight before any is used; per-thread
// sums are reduced by warp shuffles and then over the warps in warp order.  Deterministic.
constexpr int kReduceThreads = 256;
constexpr int kMaxUnitsPerReq = 1024;

__device__ __forceinline__ float4 ldcg4(const float* p) { return __ldcg(reinterpret_cast<const float4*>(p)); }

// CTA cta of ncta with NT threads; s_part holds NT / 32 * SPT floats and s_tile0 kMaxUnitsPerReq ints
// of shared memory
template <int SPT, int NT>
__device__ void reduce_tasks(const Params& P, int cta, int ncta, float* s_part, int* s_tile0) {
    constexpr int B = SPT <= 2 ? 4 : SPT == 4 ? 2 : 1;       // (unit, row group) pairs per thread in flight
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int upr = P.units_per_req, rows = P.slab_rows, rows4 = rows / 4;
    const int pairs = upr * rows4;
    const int req_items = __ldcg(P.n_items) / upr;          // items of unit 0 of every request
    // each CTA takes a contiguous range of (request, key tile) tasks; the request changes rarely inside it
    const int tasks = req_items * kItemTiles;
    const int per = (tasks + ncta - 1) / ncta;
    const int task0 = cta * per, task1 = min(tasks, task0 + per);
    int r = -1, rbeg = 0, rend = 0, N = 0;
    for (int task = task0; task < task1; ++task) {
        if (task >= rend) {
            // the request: the largest r whose first item (unit_items[r * upr].x / upr) is <= task / 2
            const int ri = task / kItemTiles;
            int lo = 0, hi = P.R;
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (__ldcg(&P.unit_items[mid * upr].x) / upr <= ri) lo = mid; else hi = mid;
            }
            r = lo;
            N = P.cu[r + 1] - P.cu[r];
            const int2 u0 = __ldcg(&P.unit_items[r * upr]);
            rbeg = (u0.x / upr) * kItemTiles;
            rend = rbeg + u0.y * kItemTiles;
            __syncthreads();                                    // the previous request's bases are no longer read
            for (int kk = threadIdx.x; kk < upr; kk += NT)
                s_tile0[kk] = __ldcg(&P.unit_items[r * upr + kk].x) * kItemTiles;
            __syncthreads();
        }
        const int tile = task - rbeg;
        if (N == 0 || tile * kTileKeys >= N) continue;     // the odd tile of a request's last item
        float acc[SPT];
#pragma unroll
        for (int s = 0; s < SPT; ++s) acc[s] = 0.f;
        for (int i0 = threadIdx.x; i0 < pairs; i0 += B * NT) {
            float4 wv[B], ev[B][SPT];
#pragma unroll
            for (int b = 0; b < B; ++b) {
                const int i = i0 + b * NT;
                bool live = i < pairs;
                size_t t = 0;
                int kk = 0, r0 = 0;
                if (live) {
                    kk = i / rows4;
                    r0 = (i - kk * rows4) * 4;
                    t = static_cast<size_t>(s_tile0[kk]) + tile;
                    live = UP_IN(t * rows + r0 + 3, P.lim_bm, P.status) &&
                           UP_IN((t * SPT + SPT - 1) * rows + r0 + 3, P.lim_be, P.status) &&
                           UP_IN(static_cast<size_t>(r * upr + kk) * rows + r0 + 3, P.lim_cvec, P.status);
                }
                if (!live) {
                    wv[b] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                    for (int sb = 0; sb < SPT; ++sb) ev[b][sb] = make_float4(0.f, 0.f, 0.f, 0.f);
                    continue;
                }
                const float4 c4 = ldcg4(P.cvec + static_cast<size_t>(r * upr + kk) * rows + r0);
                const float4 m4 = ldcg4(P.bm + t * rows + r0);
                wv[b] = make_float4(ex2(m4.x - c4.x), ex2(m4.y - c4.y), ex2(m4.z - c4.z), ex2(m4.w - c4.w));
#pragma unroll
                for (int sb = 0; sb < SPT; ++sb) ev[b][sb] = ldcg4(P.be + (t * SPT + sb) * rows + r0);
            }
#pragma unroll
            for (int b = 0; b < B; ++b)
#pragma unroll
                for (int sb = 0; sb < SPT; ++sb) {
                    const float4 w4 = wv[b], e4 = ev[b][sb];
                    acc[sb] += (e4.x * w4.x + e4.y * w4.y) + (e4.z * w4.z + e4.w * w4.w);
                }
        }
#pragma unroll
        for (int s = 0; s < SPT; ++s) {
            float x = acc[s];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
            if (lane == 0) s_part[w * SPT + s] = x;
        }
        __syncthreads();
        if (threadIdx.x < SPT) {
            const int g = tile * SPT + threadIdx.x;
            if (g * P.G < N) {
                float x = 0.f;
                for (int w2 = 0; w2 < NT / 32; ++w2) x += s_part[w2 * SPT + threadIdx.x];
                const int ne = min(P.n, N);
                if (UP_IN(P.cb[r] + g, P.nb_cap, P.status))
                    P.block_scores[P.cb[r] + g] = x * (1.0f / (static_cast<float>(ne) * P.Hq * P.G));
            }
        }
        __syncthreads();
    }
}

template <int SPT>
__global__ void __launch_bounds__(kReduceThreads) reduce_kernel(Params P) {
    pdl_wait();
    pdl_trigger();
    if (__ldcg(P.n_items + 1) == 0) return;   // plan rejected the varlen metadata
    __shared__ float s_part[kReduceThreads / 32 * SPT];
    __shared__ int s_tile0[kMaxUnitsPerReq];
    reduce_tasks<SPT, kReduceThreads>(P, blockIdx.x, gridDim.x, s_part, s_tile0);
}

// PLAN (one pass only): the kernel plans its own items (plan_prologue) instead of reading the list of
// the plan kernel.
template <int PASS, int NC, bool PLAN = false>
__global__ void __launch_bounds__(kThreads, 1)
    score_pass_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK, Params P) {
    extern __shared__ uint8_t smem_raw[];
    const Smem S = carve(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(S.full + s), 1);
            mbar_init(smem_u32(S.empty + s), kIssuers);    // one commit from each issuer
        }
        for (int b = 0; b < 4; ++b) {
            mbar_init(smem_u32(S.tfull + b), 1);
            // one arrival per epilogue warp that reads the job: 4 warps per warpgroup on it
            mbar_init(smem_u32(S.tempty + b), 4 * (PASS == 3 && NC == 4 ? 2 : job_map<PASS>(P).wpj));
        }
        mbar_init(smem_u32(S.slab_full), 1);
        mbar_init(smem_u32(S.slab_free), kIssuers);
        for (int w = 0; w < kIssuers; ++w) mbar_init(smem_u32(S.mma_done + w), 1);
        for (int w = 0; w < 2; ++w) mbar_init(smem_u32(S.tok + w), 1);
        *S.abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmQ);
        prefetch_tmap(&tmK);
    }
    // query rows that no TMA load ever writes (slab padding) must be finite: zero the slab once (a
    // planning pass uses its first kPlanScratch bytes as scratch and zeroes them after its prologue)
    for (int i = (PLAN ? kPlanScratch / 16 : 0) + threadIdx.x; i < kSlabBytes / 16; i += kThreads)
        reinterpret_cast<uint4*>(S.slab)[i] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
    if (warp == 1) {
        tmem_alloc(smem_u32(S.tmem_holder), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = static_cast<uint32_t>(uni(static_cast<int>(*S.tmem_holder)));

    // The set-up above touched only this CTA's shared memory and TMEM.  Pass 1 reads the work items its
    // predecessor (the plan kernel) writes, so every warp waits here.  Pass 2's producer and MMA warps
    // read only Q, K and the items, complete since before pass 1 ran, so they start at once; only its
    // epilogue waits, for the row normalisers of its predecessor (the merge kernel).
    if (PASS != 2) pdl_wait();
    pdl_trigger();
    int it0, it1;
    bool planned = true;
    if (PLAN) {
        int* scratch = reinterpret_cast<int*>(S.slab);
        planned = plan_prologue(P, scratch, scratch + kPlanSmemReqs, it0, it1);
        __syncthreads();                        // scratch no longer read; this CTA's item entries written
        for (int i = threadIdx.x; i < kPlanScratch / 16; i += kThreads) reinterpret_cast<uint4*>(S.slab)[i] = make_uint4(0, 0, 0, 0);
        fence_proxy_async_smem();
        __syncthreads();
    } else {
        const int n_items = uni(__ldcg(P.n_items));
        // gridDim.x = nsets * groups: CTA (set s, group g) takes the g-th share of set s's run
        const int groups = gridDim.x / P.nsets, run = n_items / P.nsets;
        const int set = blockIdx.x / groups, g = blockIdx.x % groups;
        it0 = set * run + static_cast<int>((int64_t)g * run / groups);
        it1 = set * run + static_cast<int>((int64_t)(g + 1) * run / groups);
    }

    if (warp == 0) {
        producer<NC>(P, S, &tmQ, &tmK, it0, it1);
    } else if (warp == 1 || warp >= kIssuer1Warp) {
        // warps 1 and 18 (kThreads covers exactly these and the producer and epilogue warps)
        mma_issuer<PASS, NC>(P, S, tmem_base, it0, it1, warp == 1 ? 0u : static_cast<uint32_t>(warp - kIssuer1Warp + 1));
    } else if (PASS == 3 && NC == 4) {
        switch (P.spt) {                         // blocks per key tile = 128 / G
            case 8: epilogue_one_pass_pairs<1>(P, S, tmem_base, it0, it1); break;
            case 4: epilogue_one_pass_pairs<2>(P, S, tmem_base, it0, it1); break;
            case 2: epilogue_one_pass_pairs<4>(P, S, tmem_base, it0, it1); break;
            default: epilogue_one_pass_pairs<8>(P, S, tmem_base, it0, it1); break;
        }
    } else if (PASS == 3) {
        switch (P.spt) {
            case 8: epilogue_one_pass_whole<1>(P, S, tmem_base, it0, it1); break;
            case 4: epilogue_one_pass_whole<2>(P, S, tmem_base, it0, it1); break;
            case 2: epilogue_one_pass_whole<4>(P, S, tmem_base, it0, it1); break;
            default: epilogue_one_pass_whole<8>(P, S, tmem_base, it0, it1); break;
        }
    } else {
        const JobMap jm = job_map<PASS>(P);
        switch (jm.W / 16 / jm.wpj) {            // 16-column chunks per job slice
            case 8: epilogue<PASS, 8>(P, S, tmem_base, it0, it1); break;
            case 4: epilogue<PASS, 4>(P, S, tmem_base, it0, it1); break;
            default: epilogue<PASS, 2>(P, S, tmem_base, it0, it1); break;
        }
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

// sum of parts values x[k * stride], k = 0, 1, ... in that order; the loads go out 32 at a time (the
// usual count of partials: one latency round), entries past the end add +0 and change nothing
__device__ __forceinline__ float sum_parts(const float* x, int64_t stride, int parts) {
    constexpr int kBatch = 32;
    float s = 0.f;
    for (int k = 0; k < parts; k += kBatch) {
        float v[kBatch];
#pragma unroll
        for (int i = 0; i < kBatch; ++i) v[i] = k + i < parts ? __ldcg(x + (size_t)(k + i) * stride) : 0.f;
#pragma unroll
        for (int i = 0; i < kBatch; ++i) s += v[i];
    }
    return s;
}

__global__ void finalize_kernel(Params P) {
    pdl_wait();
    pdl_trigger();
    if (__ldcg(P.n_items + 1) == 0) return;   // plan rejected the varlen metadata
    const int parts = P.units_per_req * 4;       // (unit, warpgroup) partials, summed in a fixed order
    const int nb_total = P.cb[P.R];
    const int stride = gridDim.x * blockDim.x;
    for (int gb = blockIdx.x * blockDim.x + threadIdx.x; gb < nb_total; gb += stride) {
        const int r = find_segment(P.cb, P.R, gb);
        const int ne = min(P.n, P.cu[r + 1] - P.cu[r]);
        if (!UP_IN(gb + (int64_t)(parts - 1) * P.nb_cap, P.lim_blk, P.status) || !UP_IN(gb, P.nb_cap, P.status)) continue;
        P.block_scores[gb] = sum_parts(P.blk + gb, P.nb_cap, parts) * (1.0f / (static_cast<float>(ne) * P.Hq * P.G));
    }
    if (P.token_scores != nullptr) {
        for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < P.T; t += stride) {
            const int r = find_segment(P.cu, P.R, t);
            const int ne = min(P.n, P.cu[r + 1] - P.cu[r]);
            if (!UP_IN(t + (int64_t)(parts - 1) * P.T, P.lim_tok, P.status)) continue;
            P.token_scores[t] = sum_parts(P.tok + t, P.T, parts) * (1.0f / (static_cast<float>(ne) * P.Hq));
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
    const cudaError_t e = launch_pdl(score_pass_kernel<PASS, NC>, dim3(grid), dim3(kThreads), kSmemBytes, st, q, k, P);
    count_launch();
    return e;
}

static cudaError_t launch_merge(const Params& P, int64_t merge_rows, cudaStream_t st) {
    const int mgrid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(cdiv(merge_rows, 8), 16 * num_sms())));
    const cudaError_t e = launch_pdl(merge_kernel, dim3(mgrid), dim3(256), 0, st, P);
    count_launch();
    return e;
}

// two passes (row statistics, merge, recompute with the column sums); finalize follows
template <int NC>
static cudaError_t launch_both(const CUtensorMap& q, const CUtensorMap& k, const Params& P, int grid,
                               int64_t merge_rows, cudaStream_t st) {
    cudaError_t e = launch_pass<1, NC>(q, k, P, grid, st);
    if (e != cudaSuccess) return e;
    e = launch_merge(P, merge_rows, st);
    if (e != cudaSuccess) return e;
    return launch_pass<2, NC>(q, k, P, grid, st);
}

// one pass (row statistics and block sums), merge, reduce into the block scores; plan_inside: the pass
// plans its own items (no plan kernel before it)
template <int NC>
static cudaError_t launch_one(const CUtensorMap& q, const CUtensorMap& k, const Params& P, int grid,
                              int64_t merge_rows, int64_t req_tiles, cudaStream_t st, bool plan_inside = false) {
    cudaError_t e;
    if (plan_inside) {
        static std::once_flag once;
        static cudaError_t attr = cudaSuccess;
        std::call_once(once, [] {
            attr = cudaFuncSetAttribute(score_pass_kernel<3, NC, true>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        });
        if (attr != cudaSuccess) return attr;
        e = launch_pdl(score_pass_kernel<3, NC, true>, dim3(grid), dim3(kThreads), kSmemBytes, st, q, k, P);
        count_launch();
    } else {
        e = launch_pass<3, NC>(q, k, P, grid, st);
    }
    if (e != cudaSuccess) return e;
    e = launch_merge(P, merge_rows, st);
    if (e != cudaSuccess) return e;
    const int rgrid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(req_tiles, 8 * num_sms())));
    switch (P.spt) {
        case 8: e = launch_pdl(reduce_kernel<8>, dim3(rgrid), dim3(kReduceThreads), 0, st, P); break;
        case 4: e = launch_pdl(reduce_kernel<4>, dim3(rgrid), dim3(kReduceThreads), 0, st, P); break;
        case 2: e = launch_pdl(reduce_kernel<2>, dim3(rgrid), dim3(kReduceThreads), 0, st, P); break;
        default: e = launch_pdl(reduce_kernel<1>, dim3(rgrid), dim3(kReduceThreads), 0, st, P); break;
    }
    count_launch();
    return e;
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
    if (G != 16 && G != 32 && G != 64 && G != 128) return 0;
    return layout(R, T, g, Hkv, nb_cap, with_token_scores != 0, G).total;
}

extern "C" up_status up_score_blocks(const uint16_t* Q, const uint16_t* K, const int32_t* cu_seqlens, int R,
                                     int64_t T, int Hq, int Hkv, int dk, int G, int n, float sm_scale,
                                     const int32_t* cu_blocks, int64_t nb_cap, float* block_scores,
                                     float* token_scores, void* ws, size_t ws_bytes, int32_t* dev_status,
                                     void* stream) {
    // Q and K may be NULL for a batch without tokens (T = 0): nothing is read from them
    if ((T > 0 && (!Q || !K)) || !cu_seqlens || !cu_blocks || !block_scores || !ws || !dev_status) return UP_ERR_ARG;
    if (R <= 0 || T < 0 || T >= (int64_t(1) << 31) || nb_cap < 0 || !(sm_scale > 0.f) || !isfinite(sm_scale))
        return UP_ERR_ARG;
    Geometry g;
    if (!geometry(Hq, Hkv, dk, n, &g)) return UP_ERR_SHAPE;
    if (G != 16 && G != 32 && G != 64 && G != 128) return UP_ERR_SHAPE;
    if (!aligned16(Q) || !aligned16(K) || !aligned16(ws)) return UP_ERR_SHAPE;
    const Layout L = layout(R, T, g, Hkv, nb_cap, token_scores != nullptr, G);
    // one tcgen05 pass unless per-token scores are asked for (they need the recompute pass)
    const bool one_pass = token_scores == nullptr && one_pass_ok(g.J) && Hkv * g.slabs <= kMaxUnitsPerReq;
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
    P.wide2 = g.J == 2 ? 1 : 0;
    P.box_rows = g.box_rows;
    P.units_per_req = Hkv * g.slabs;
    P.a = sm_scale * 1.4426950408889634f;
    P.nb_cap = nb_cap;
    P.items = reinterpret_cast<int4*>(w + L.items);
    P.unit_items = reinterpret_cast<int2*>(w + L.unit_items);
    P.n_items = reinterpret_cast<int*>(w + L.n_items);
    P.ml = reinterpret_cast<float2*>(w + L.ml);
    P.cvec = reinterpret_cast<float*>(w + L.cvec);
    P.blk = reinterpret_cast<float*>(w + L.blk);
    P.tok = token_scores ? reinterpret_cast<float*>(w + L.tok) : nullptr;
    P.be = one_pass ? reinterpret_cast<float*>(w + L.be) : nullptr;
    P.bm = one_pass ? reinterpret_cast<float*>(w + L.bm) : nullptr;
    P.spt = kTileKeys / G;
    P.lim_items = L.items_cap;
    P.lim_units = L.units;
    P.lim_ml = L.items_cap * g.slab_rows;
    P.lim_cvec = L.units * g.slab_rows;
    P.lim_blk = static_cast<int64_t>(Hkv) * g.slabs * 4 * nb_cap;
    P.lim_tok = token_scores ? static_cast<int64_t>(Hkv) * g.slabs * 4 * T : 0;
    P.lim_be = one_pass ? L.items_cap * kItemTiles * (kTileKeys / G) * g.slab_rows : 0;
    P.lim_bm = one_pass ? L.items_cap * kItemTiles * g.slab_rows : 0;
    P.block_scores = block_scores;
    P.token_scores = token_scores;
    P.status = dev_status;
    P.nsets = work_sets(P.units_per_req, g.slabs, num_sms());

    // the one pass with at most kPlanSmemReqs requests plans inside its own launch
    if (T > 0 && one_pass && R <= kPlanSmemReqs) {
        CUtensorMap tq, tk;
        if (!make_map(&tq, Q, T, Hq, dk, g.box_rows) || !make_map(&tk, K, T, Hkv, dk, kTileKeys)) return UP_ERR_CUDA;
        int grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(num_sms(), L.items_cap)));
        grid = grid / P.nsets * P.nsets;
        const int64_t merge_rows = L.units * g.slab_rows;
        const int64_t req_tiles = L.items_cap / P.units_per_req * kItemTiles;
        cudaError_t e;
        switch (g.nc) {
            case 1: e = launch_one<1>(tq, tk, P, grid, merge_rows, req_tiles, st, true); break;
            case 2: e = launch_one<2>(tq, tk, P, grid, merge_rows, req_tiles, st, true); break;
            default: e = launch_one<4>(tq, tk, P, grid, merge_rows, req_tiles, st, true); break;
        }
        return e == cudaSuccess ? UP_OK : UP_ERR_CUDA;
    }
    // the item list by a grid of CTAs (one while the requests' offsets do not fit their shared memory)
    const int pgrid = R <= kPlanSmemReqs
                          ? static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(cdiv(L.items_cap, kPlanThreads), num_sms())))
                          : 1;
    cudaError_t le = launch_pdl(plan_kernel, dim3(pgrid), dim3(kPlanThreads), 0, st, P);
    count_launch();
    if (le != cudaSuccess) return UP_ERR_CUDA;
    if (T > 0) {
        CUtensorMap tq, tk;
        if (!make_map(&tq, Q, T, Hq, dk, g.box_rows) || !make_map(&tk, K, T, Hkv, dk, kTileKeys)) return UP_ERR_CUDA;
        int grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(num_sms(), L.items_cap)));
        grid = grid / P.nsets * P.nsets;
        cudaError_t e;
        const int64_t merge_rows = L.units * g.slab_rows;
        if (one_pass) {
            const int64_t req_tiles = L.items_cap / P.units_per_req * kItemTiles;
            switch (g.nc) {
                case 1: e = launch_one<1>(tq, tk, P, grid, merge_rows, req_tiles, st); break;
                case 2: e = launch_one<2>(tq, tk, P, grid, merge_rows, req_tiles, st); break;
                default: e = launch_one<4>(tq, tk, P, grid, merge_rows, req_tiles, st); break;
            }
            return e == cudaSuccess ? UP_OK : UP_ERR_CUDA;
        }
        switch (g.nc) {
            case 1: e = launch_both<1>(tq, tk, P, grid, merge_rows, st); break;
            case 2: e = launch_both<2>(tq, tk, P, grid, merge_rows, st); break;
            default: e = launch_both<4>(tq, tk, P, grid, merge_rows, st); break;
        }
        if (e != cudaSuccess) return UP_ERR_CUDA;
    }
    const int fgrid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(4 * num_sms(), cdiv(std::max<int64_t>(nb_cap, T), 256))));
    le = launch_pdl(finalize_kernel, dim3(fgrid), dim3(256), 0, st, P);
    count_launch();
    return le == cudaSuccess ? UP_OK : UP_ERR_CUDA;
}
