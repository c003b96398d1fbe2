/*
 * uniprefill.h - C ABI of libuniprefill.so, the GB300 (sm_103a) hot path of
 * UniPrefill's block-wise dynamic token dropping at one full-attention layer.
 *
 * Source: "UniPrefill: Universal Long-Context Prefill Acceleration via
 * Block-wise Dynamic Sparsification" (arXiv 2605.06221), cited as [UP ...].
 *
 * One drop step over a varlen packed batch:
 *   up_score_blocks  S = Q[N-n:N] K^T / sqrt(d_k) -> two-pass online softmax -> block mass   [UP 3.2, Eqs. 2-4, 13]
 *   up_select_topp   packed (score,index) keys, descending sort, top-p prefix, forced tokens [UP 3.3 Eq. 5, 3.5 Eq. 14]
 *   up_compact       stable gather of the kept tokens + query_start_loc / seq_lens / history [UP 3.5]
 *   up_scatter_back  write the kept rows' new states into the full-length residual         [UP 3.4, Eq. 8]
 *   up_slot_mapping  KV slot ids of a (compacted) stream from a layer's block table         [UP 3.5, Eq. 16]
 *   up_seqused       per-layer KV length seen by decode, from the drop history              [UP 3.5, Eq. 17]
 *
 * Conventions shared by every call:
 *  - All array pointers are DEVICE pointers owned by the caller; the library
 *    never allocates, frees or keeps a pointer after a call returns.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  Every
 *    call only enqueues kernels on it and returns without synchronising,
 *    except up_read_status, which synchronises the stream.
 *  - bf16 tensors are passed as uint16_t bit patterns, row-major, packed over
 *    the tokens of all requests: token t of request r is row cu_seqlens[r]+t.
 *  - cu_seqlens is int32 [R+1], cu_seqlens[0] = 0, non-decreasing,
 *    cu_seqlens[R] = T.  Requests may be empty.  (vLLM's query_start_loc.)
 *  - cu_blocks is int32 [R+1], the exclusive scan of ceil(N_r / G); block g
 *    of request r lives at index cu_blocks[r] + g (see up_make_cu_blocks).
 *  - Errors found on the host (bad scalars, NULL pointers, misalignment,
 *    workspace too small) are returned before anything is launched.  Errors
 *    that need the device's data (a malformed cu_seqlens, a request with too
 *    many blocks, a position outside the block table, an internal wait that
 *    ran out) are recorded in the caller's int32 `dev_status` word (first
 *    error wins, 0 = no error); the kernels then skip their work and return.
 *    No kernel traps, asserts or waits without a bound.  Read the word with
 *    up_read_status.  Clear it (to 0) yourself before reusing it.
 *  - Results are deterministic: the same inputs give bit-identical outputs
 *    run to run, whatever the packing of the other requests.
 *  - Calls are stateless and may run concurrently on different streams with
 *    different workspaces.
 */
#ifndef UNIPREFILL_H
#define UNIPREFILL_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    UP_OK = 0,
    UP_ERR_ARG = 1,        /* NULL pointer or scalar out of range                            */
    UP_ERR_SHAPE = 2,      /* unsupported geometry (d_k, G, n, head ratio, hidden, alignment) */
    UP_ERR_WORKSPACE = 3,  /* ws_bytes smaller than the *_workspace_bytes query              */
    UP_ERR_CUDA = 4,       /* a CUDA runtime call or kernel launch failed                    */
    UP_ERR_DEVICE = 5      /* returned by up_read_status when dev_status holds an error      */
} up_status;

/* device status codes written to `dev_status` */
#define UP_DEV_OK               0
#define UP_DEV_BAD_CU_SEQLENS   1   /* cu_seqlens not 0..T non-decreasing                         */
#define UP_DEV_BAD_CU_BLOCKS    2   /* cu_blocks inconsistent with cu_seqlens and G, or > nb_cap  */
#define UP_DEV_TOO_MANY_BLOCKS  3   /* a request over UP_MAX_BLOCKS_PER_REQUEST blocks, no select ws */
#define UP_DEV_WAIT_TIMEOUT     4   /* a pipeline wait inside a kernel ran past its time bound    */
#define UP_DEV_BAD_POSITION     5   /* Eq. 16: a position beyond its block-table row (slot = -1) */
#define UP_DEV_BAD_TOKEN_COUNT  6   /* num_actual_tokens outside [0, T_upper]                     */
#define UP_DEV_BOUNDS           7   /* bounds-checked build only: an index outside its array      */

#define UP_MAX_BLOCKS_PER_REQUEST 8192   /* up to this many blocks up_select_topp sorts a request in
                                            shared memory; longer requests need its workspace */

/* ------------------------------------------------------------------------------------------- */
/* sizing helpers (host only, no CUDA call)                                                     */

/* Upper bound of sum_r ceil(N_r / G) for any split of T tokens into R requests: T / G + R. */
int64_t up_max_blocks(int R, int64_t T, int G);

/* Workspace of up_score_blocks; 0 when the arguments are invalid.  nb_cap is the length of the
 * caller's block arrays (>= cu_blocks[R]); with_token_scores != 0 reserves the per-token
 * partials needed when token_scores is requested. */
size_t up_score_workspace_bytes(int R, int64_t T, int Hq, int Hkv, int dk, int G, int n,
                                int64_t nb_cap, int with_token_scores);

/* Workspace of up_compact. */
size_t up_compact_workspace_bytes(int R, int64_t T);

/* Workspace of up_select_topp for block arrays of nb_cap entries (two key arrays of nb_cap uint64). */
size_t up_select_workspace_bytes(int64_t nb_cap);

/* One workspace big enough for every call of a drop step (score with token scores, select, compact),
 * which run one after another on a stream and may therefore share it. */
size_t up_workspace_bytes(int R, int64_t T, int Hq, int Hkv, int dk, int G, int n, int64_t nb_cap);

/* ------------------------------------------------------------------------------------------- */
/* the drop step                                                                                */

/* cu_blocks[r+1] = cu_blocks[r] + ceil((cu_seqlens[r+1] - cu_seqlens[r]) / G), cu_blocks[0] = 0
 * (the block partition B_g of [UP 3.2, text before Eq. 4]).  cu_blocks: int32 [R+1]. */
up_status up_make_cu_blocks(const int32_t* cu_seqlens, int R, int64_t T, int G,
                            int32_t* cu_blocks, int32_t* dev_status, void* stream);

/* Block scores b_g of [UP 3.2, Eq. 4] (the "o -> b" half of Eq. 13), for every request:
 *   for query heads h, window rows j in [N-n_eff, N) (n_eff = min(n, N)), keys i <= j:
 *     A_{h,j,i} = softmax_i(q_{h,j} . k_{kv(h),i} * sm_scale)          [UP Eq. 2, causal in the window]
 *     s_i  = 1/(n_eff * Hq) * sum_h sum_j A_{h,j,i}                    [UP Eq. 3, mean over heads]
 *     b_g  = 1/G * sum_{i in B_g} s_i     (B_g = {gG .. min((g+1)G, N)-1}; the last block is
 *                                          still divided by G)         [UP Eq. 4]
 *   kv(h) = h / (Hq / Hkv).  The softmax normalises over the complete key range before any
 *   block reduction, in two passes [UP 3.5 "Kernel design"]: one pass over S gives each row's
 *   maximum and sum and its sums over every block against a running maximum, and the second pass
 *   runs over those block sums with the row normalisers (with token_scores, the second pass
 *   recomputes S instead).  S is never materialised.
 * Q: bf16 [T, Hq, dk] (only each request's last n rows are read); K: bf16 [T, Hkv, dk]; both may
 * be NULL when T = 0.
 * Both 16-byte aligned.  dk in {64, 128, 256}; Hq % Hkv == 0; G in {16, 32, 64, 128};
 * n in {16, 32, 64, 128} or a multiple of 128 up to 1024.  sm_scale is usually 1/sqrt(dk).
 * block_scores: fp32 [nb_cap] (entries cu_blocks[r] .. cu_blocks[r+1]-1 written).
 * token_scores: optional fp32 [T] (s_i; NULL to skip).
 * Arithmetic: bf16 products, fp32 accumulation (tcgen05 tensor cores), fp32 softmax.
 * ws: device workspace of up_score_workspace_bytes(...) bytes, no initialisation needed. */
up_status up_score_blocks(const uint16_t* Q, const uint16_t* K, const int32_t* cu_seqlens,
                          int R, int64_t T, int Hq, int Hkv, int dk, int G, int n, float sm_scale,
                          const int32_t* cu_blocks, int64_t nb_cap,
                          float* block_scores, float* token_scores,
                          void* ws, size_t ws_bytes, int32_t* dev_status, void* stream);

/* Top-p selection [UP 3.3, Eq. 5] with the packed sort key of [UP 3.5, Eq. 14], per request:
 *   key_g = (phi(b_g) << 32) | g as uint64, phi(x) = bits(x) ^ 0x80000000 for x >= 0;
 *   the keys are radix-sorted descending (equal scores: higher g first);
 *   k* = min k with sum_{first k} b >= p * sum_g b  (sums in fp64);
 *   token_keep_i = [block(i) among the first k*] or i < A (sinks) or i >= N - n (window);
 *   block_keep_g = any token of B_g kept.
 * block_scores: fp32 [nb_cap], finite and >= 0.  p in (0, 1]; A >= 0; n >= 1; G a power of two.
 * block_keep: u8 [nb_cap]; token_keep: u8 [T], 16-byte aligned (it is written with 16-byte stores;
 * a misaligned pointer returns UP_ERR_SHAPE; may be NULL when T = 0); kstar: int32 [R] (0 for empty
 * requests).
 * ws: device workspace of up_select_workspace_bytes(nb_cap) bytes, 16-byte aligned, no initialisation
 * needed, or NULL.  A request of at most UP_MAX_BLOCKS_PER_REQUEST blocks is sorted in shared memory and
 * never touches it; a longer request sorts its keys through it (the same stable passes in tiles of 8192
 * keys), and without it sets UP_DEV_TOO_MANY_BLOCKS.  A non-NULL ws that is smaller or misaligned
 * returns UP_ERR_WORKSPACE before any launch. */
up_status up_select_topp(const float* block_scores, const int32_t* cu_blocks,
                         const int32_t* cu_seqlens, int R, int64_t T, int64_t nb_cap,
                         int G, int n, int A, double p,
                         uint8_t* block_keep, uint8_t* token_keep, int32_t* kstar,
                         void* ws, size_t ws_bytes, int32_t* dev_status, void* stream);

/* Compaction and metadata patch [UP 3.5 "vLLM scheduler integration"]:
 * kept tokens (token_keep != 0) are gathered in ascending packed order (stable), T' of them:
 *   kept_index[k]     = packed index of the k-th kept token, int32 [T] (first T' written)
 *   out_hidden[k, :]  = hidden[kept_index[k], :]  (bf16 [T, hdim]; optional with hidden)
 *   out_positions[k]  = positions[kept_index[k]]  (int64; optional with positions)
 *   out_slots[k]      = slots[kept_index[k]]      (int64; optional with slots)
 *   new_cu_seqlens    = the patched query_start_loc, int32 [R+1]
 *   new_seq_lens[r]   = kept tokens of request r, int32 [R]
 *   num_actual_tokens = T', int32 [1] (stays on the device; buffers are sized by T)
 *   kept_len[layer*R + r] = new_seq_lens[r] and drop_layer[layer] = 1 record the drop history
 *   {(l_k, s_k^r)} of [UP 3.5] (both optional; kept_len int32 [L, R], drop_layer u8 [L]).
 * hdim % 8 == 0; hidden/out_hidden 16-byte aligned; token_keep 16-byte aligned (may be NULL when
 * T = 0, as may hidden/positions/slots and their outputs).
 * cu_seqlens that is not a non-decreasing 0..T sequence sets UP_DEV_BAD_CU_SEQLENS in dev_status and
 * num_actual_tokens = 0, and leaves new_cu_seqlens, new_seq_lens and the drop history unwritten;
 * kept_index and the gathered rows, which do not depend on cu_seqlens, are still written.
 * ws: up_compact_workspace_bytes(R, T) bytes. */
up_status up_compact(const uint8_t* token_keep, const int32_t* cu_seqlens, int R, int64_t T,
                     const uint16_t* hidden, int hdim, const int64_t* positions, const int64_t* slots,
                     uint16_t* out_hidden, int64_t* out_positions, int64_t* out_slots,
                     int32_t* kept_index, int32_t* new_cu_seqlens, int32_t* new_seq_lens,
                     int32_t* num_actual_tokens, int32_t* kept_len, uint8_t* drop_layer,
                     int L, int layer, void* ws, size_t ws_bytes, int32_t* dev_status, void* stream);

/* up_compact without a workspace argument.  The paper has no counterpart: this entry point exists for
 * callers that cannot allocate or lend device scratch memory (an engine whose memory planner owns all
 * device memory after start-up, a plugin host that only passes the tensors it already holds, a loop
 * that must avoid cudaMalloc's implicit synchronisation).  Arguments and results are those of
 * up_compact, minus ws/ws_bytes.  Its per-tile counts and offsets live in a fixed array inside the
 * library's device image (2 * (UP_NOALLOC_MAX_TOKENS / 1024 + 1) int32, about 128 KB), present on every
 * GPU that loads the library until the process exits; the call allocates nothing.
 *  - T > UP_NOALLOC_MAX_TOKENS returns UP_ERR_WORKSPACE before any launch (use up_compact instead).
 *  - The first call on a device looks up the array's device address (cudaGetSymbolAddress) with that
 *    device current; make that first call before any stream capture.  The address is kept for the
 *    rest of the process: after cudaDeviceReset on that device the entry point must not be called
 *    again (the library's device image, and with it the array, may have moved).
 *  - Every call on a device shares the one array and leaves its contents behind (nothing in it needs
 *    clearing: each call overwrites what it reads).  Calls whose kernels can overlap on the GPU (for
 *    example on two streams without ordering between them) race on it and give wrong results; order
 *    them on one stream or use up_compact with separate workspaces. */
#define UP_NOALLOC_MAX_TOKENS (16384 * 1024)
up_status up_compact_noalloc(const uint8_t* token_keep, const int32_t* cu_seqlens, int R, int64_t T,
                             const uint16_t* hidden, int hdim, const int64_t* positions, const int64_t* slots,
                             uint16_t* out_hidden, int64_t* out_positions, int64_t* out_slots,
                             int32_t* kept_index, int32_t* new_cu_seqlens, int32_t* new_seq_lens,
                             int32_t* num_actual_tokens, int32_t* kept_len, uint8_t* drop_layer,
                             int L, int layer, int32_t* dev_status, void* stream);

/* End-of-block carry-forward [UP 3.4, Eq. 8], in place:
 *   residual[kept_index[k], :] = new_states[k, :]  for k < *num_actual_tokens;
 *   rows of dropped tokens are not touched (they keep H^(b,0)).
 * new_states: bf16 [T_upper, hdim], the compacted stream (T_upper >= *num_actual_tokens; a larger
 * count is reported as UP_DEV_BAD_TOKEN_COUNT and nothing is copied); residual: bf16 [T, hdim], the
 * full-length stream that up_compact compacted (every kept_index entry is below T); both 16-byte
 * aligned (with T_upper = 0 nothing is read or written and every pointer may be NULL);
 * hdim % 8 == 0.  kept_index/num_actual_tokens as produced by up_compact over that stream. */
up_status up_scatter_back(const uint16_t* new_states, const int32_t* kept_index,
                          const int32_t* num_actual_tokens, int64_t T_upper, int hdim,
                          uint16_t* residual, int32_t* dev_status, void* stream);

/* KV slot mapping of a layer [UP 3.5, Eq. 16]:
 *   slot_t = block_table[r_t * max_blocks + floor(p_t / B)] * B + (p_t mod B)
 * r_t = the request of token t under cu_seqlens (e.g. the compacted new_cu_seqlens), p_t =
 * positions[t] (int64).  Tokens t < *num_tokens (or < T_upper if num_tokens is NULL).
 * block_table: int32 [R, max_blocks]; slots: int64 [T_upper] (positions and slots may be NULL
 * when T_upper = 0).  A position outside
 * [0, max_blocks*B) writes -1 and sets UP_DEV_BAD_POSITION. */
up_status up_slot_mapping(const int64_t* positions, const int32_t* cu_seqlens, int R, int64_t T_upper,
                          const int32_t* num_tokens, const int32_t* block_table, int max_blocks, int B,
                          int64_t* slots, int32_t* dev_status, void* stream);

/* KV length visible to layer `layer` during decode [UP 3.5, Eq. 17]:
 *   seqused_r = kept_len[l- * R + r] + (kv_len_r - orig_len_r),
 *   l- = max { l < layer : drop_layer[l] != 0 };  with no such l: seqused_r = kv_len_r.
 * kept_len: int32 [L, R]; drop_layer: u8 [L]; orig_len, kv_len, seqused: int32 [R]. */
up_status up_seqused(const int32_t* kept_len, const uint8_t* drop_layer, int L, int R, int layer,
                     const int32_t* orig_len, const int32_t* kv_len, int32_t* seqused, void* stream);

/* ------------------------------------------------------------------------------------------- */
/* status and introspection                                                                     */

/* Synchronises `stream`, copies *dev_status to *host_out, returns UP_ERR_DEVICE if it is not 0. */
up_status up_read_status(const int32_t* dev_status, int32_t* host_out, void* stream);

/* Static strings for an up_status (codes 0..5) or, with device != 0, a UP_DEV_* code. */
const char* up_status_string(int code, int device);

/* Number of kernels this library has launched in this process (for launch accounting). */
uint64_t up_kernel_launches(void);

/* ABI version of this header: 2 (up_select_topp takes a workspace). */
int up_abi_version(void);

/* 1 in the bounds-checked build of the library (compiled with -DUP_DEBUG_BOUNDS, a development aid:
 * every kernel checks each global index against its array's length, records UP_DEV_BOUNDS in the
 * status word on a violation and skips the access), 0 in the normal build. */
int up_debug_bounds(void);

#ifdef __cplusplus
}
#endif
#endif /* UNIPREFILL_H */
