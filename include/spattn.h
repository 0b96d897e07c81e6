/*
 * spattn.h -- C ABI of the block-sparse masked attention library (libspattn.so).
 *
 * The library computes the forward pass of masked scaled-dot-product attention
 * under structured sparse masks on one NVIDIA B300 (sm_103a):
 *
 *     y_i   = sum_{j in S_i} alpha_ij v_j,
 *     alpha_ij = exp(scale q_i.k_j) / sum_{l in S_i} exp(scale q_i.k_l),
 *     LSE_i = ln sum_{j in S_i} exp(scale q_i.k_j)
 *
 * with the softmax normalised over the allowed set S_i only ("Sparse attention"
 * glossary, glossary.selfmadequant.com, section "Choose the available reads", the
 * displayed equation for y_i and alpha_ij).  S_i is a union of simple rules
 * ("Attention variants", sreshtalluri.github.io, section 4 "Build it from
 * scratch": causal, sliding_window, local_strided, with_global), intersected with
 * causality when the mask is causal.  All indices are 0-based.
 *
 * Conventions for every call:
 *   - Every function returns a spattn_status; nothing throws or exits across the
 *     ABI.  spattn_last_error() gives a message for the last failure on the
 *     calling thread.
 *   - Device pointers are CUDA device addresses on the current device; the caller
 *     owns them.  Q, K, V and O are [B, H, T, d] contiguous row-major tensors of the
 *     input dtype, 16-byte aligned; LSE is [B, H, T] fp32.
 *   - `cuda_stream` is a cudaStream_t (NULL = the legacy default stream).
 *   - A plan is reusable across B, H, dtypes and calls (the mask is shared by all
 *     batches and heads, as create_block_mask(..., B=None, H=None) shares it in
 *     "Attention variants", section "Use the library").  Distinct plans may be used
 *     concurrently from different threads; one plan must not be used by two
 *     concurrent spattn_fwd calls (it owns the packing scratch they would share).
 */
#ifndef SPATTN_H_
#define SPATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SPATTN_OK = 0,
  SPATTN_ERR_INVALID_SPEC = 1, /* mask fields outside their domain            */
  SPATTN_ERR_SHAPE = 2,        /* T, d, B, H or a capacity out of range        */
  SPATTN_ERR_DTYPE = 3,        /* dtype not supported for this head dim        */
  SPATTN_ERR_ALIGN = 4,        /* a device pointer is not 16-byte aligned      */
  SPATTN_ERR_NULL = 5,         /* a required pointer is NULL                   */
  SPATTN_ERR_CUDA = 6,         /* a CUDA runtime / driver call failed          */
  SPATTN_ERR_TIMEOUT = 7,      /* a device-side wait ran out of its time budget */
  SPATTN_ERR_UNSUPPORTED = 8   /* valid request this build does not implement  */
} spattn_status;

typedef enum { SPATTN_BF16 = 0, SPATTN_FP32 = 1 } spattn_dtype;

/*
 * Mask specification.  Allowed pairs (i, j), 0 <= i, j < T, with d = dilation:
 *   causal = 1:  j <= i and ((i-j) % d == 0 and (i-j < window*d or window == 0)
 *                 or j strided or j global or i global or (i, j) random)
 *   causal = 0:  (|i-j| % d == 0 and (|i-j| <= radius*d or radius == -1))
 *                 or j strided or j global or i global or (i, j) random
 * where "j strided" means stride > 0 and j % stride == stride_offset, "global"
 * means a member of global_pos, and "(i, j) random" means the pair
 * (i / rand_block, j / rand_block) is listed in rand_pairs.
 * Sources: window counts the query itself (glossary, "Choose the available
 * reads": S_i = {max(1,i-w+1),...,i}); window 0 is the full causal triangle and
 * strided columns are read by every later query (octlm.ramaa.tech "Sparse
 * attention", section "One mask function for every pattern"); stride_offset 0 is
 * that page's j % s == 0, stride-1 is local_strided's j % s == s-1 ("Attention
 * variants", section 4); a bidirectional radius r reads 2r+1 keys ("Attention
 * variants", section 3, "local radius 2": query 12 reads 10..14); global rows
 * read every key and global columns are read by every query, and both stay
 * causal in a causal mask (with_global and the look-ahead warning after it).
 * A dilation d > 1 keeps every d-th key of the local window, so a causal window
 * reads i, i-d, ..., i-(window-1)d ("Attention variants", section 6, the
 * dilated(n, w, d) exercise: gap >= 0, gap % d == 0, gap < w d); d = 0 or 1 is the
 * contiguous window.
 * Domains: causal in {0,1}; causal: window >= 0 and radius == -1; bidirectional:
 * radius >= -1 and window == 0; stride >= 0; 0 <= stride_offset < stride (or 0
 * when stride == 0); 0 <= n_global <= T; global_pos is a HOST array of n_global
 * distinct positions in [0, T), any order (it is copied; the caller keeps
 * ownership); 0 <= dilation <= 2^31, and with dilation > 1 window and radius at
 * most 2^31.  Random blocks (BigBird's random connections, "Sparse and
 * sliding-window attention", section "Block-sparse attention: BigBird"): n_rand
 * >= 0 pairs (query block, key block) in a HOST array rand_pairs[2 * n_rand], any
 * order, distinct, each block index in [0, ceil(T / rand_block)); rand_block one of
 * 16, 32, 64, 128 when n_rand > 0 (ignored otherwise).  Which blocks are random is
 * the caller's draw: the library takes the list as given.  Anything else is
 * SPATTN_ERR_INVALID_SPEC.
 */
typedef struct {
  int32_t causal;
  int64_t window;
  int64_t radius;
  int64_t stride;
  int64_t stride_offset;
  int32_t n_global;
  const int32_t* global_pos;
  int64_t dilation;
  int32_t rand_block;
  int64_t n_rand;
  const int32_t* rand_pairs;
} spattn_mask_spec;

typedef struct spattn_plan spattn_plan; /* opaque, owned by the library */

/* Validate a mask spec for sequence length T on the host only (no CUDA call).
 * Same rules as spattn_plan_create.  SPATTN_OK or SPATTN_ERR_INVALID_SPEC /
 * SPATTN_ERR_SHAPE (T < 1 or T > 2^30) / SPATTN_ERR_NULL. */
spattn_status spattn_mask_validate(const spattn_mask_spec* spec, int64_t T);

/*
 * Build the block-sparse plan of a mask for sequence length T and head dim
 * head_dim (64 or 128) on the current device.  The plan is the compiled block
 * mask of "Attention variants" (section "Use the library": create_block_mask,
 * "never loading zero blocks"): every (query block, key block) tile of the
 * BM x BN = 128 x 128 grid is classified empty / full / partial from an exact
 * per-tile count of allowed pairs; strided and global key columns outside each
 * query group's band are compacted into a dense column list; and the execution
 * schedule walks only non-empty work.  Kernels run on `cuda_stream`; the call is
 * synchronous on return.  *out receives a new plan (free with
 * spattn_plan_destroy).  Errors: NULL, INVALID_SPEC, SHAPE (T out of range or
 * head_dim not 64/128), CUDA.
 */
spattn_status spattn_plan_create(const spattn_mask_spec* spec, int64_t T, int32_t head_dim,
                                 void* cuda_stream, spattn_plan** out);

/* Totals of the natural 128 x 128 grid: allowed pairs per (batch, head) (the
 * glossary's edge count E, "When the cost is linear"), tile class counts, and
 * the tile sizes.  Any output pointer may be NULL. */
spattn_status spattn_plan_info(const spattn_plan* plan, int64_t* pairs_per_head,
                               int64_t* n_full, int64_t* n_partial, int64_t* n_empty,
                               int32_t* bm, int32_t* bn);

/* Copy the non-empty tiles of the natural grid to HOST arrays, in canonical order
 * (qb ascending, then kb ascending): query block, key block, exact allowed-pair
 * count, class (1 = full: every cell of the tile inside [0,T)^2 is allowed;
 * 2 = partial).  `cap` is the capacity of each array; *n receives the number of
 * non-empty tiles (if *n > cap only cap entries are written and the call returns
 * SPATTN_ERR_SHAPE).  Any of qb/kb/cnt/cls may be NULL to skip it. */
spattn_status spattn_plan_copy_tiles(const spattn_plan* plan, int32_t* qb, int32_t* kb,
                                     int32_t* cnt, uint8_t* cls, int64_t cap, int64_t* n);

/* Copy the compacted sparse-column list C = sorted(strided columns U global
 * columns) to a HOST array (same capacity rules as spattn_plan_copy_tiles). */
spattn_status spattn_plan_copy_columns(const spattn_plan* plan, int32_t* cols, int64_t cap,
                                       int64_t* n);

/*
 * Execution schedule the forward kernels walk, copied to HOST arrays.
 * which = 0: the bf16 tensor-core kernel (groups of 256 query rows = two 128-row
 * query tiles); which = 1: the fp32 kernel (groups of 64 rows); which = 2: the bf16
 * kernel's schedule over the residue classes of a dilated window (used instead of 0
 * when dilation d > 1, there are no strided or global columns and d divides T: class
 * r holds positions r, r+d, ..., where the window is contiguous; empty otherwise).
 * items:   4 int32 per work item  {q_row0, entry_offset, entry_count, flags}
 *          flags bit 0: rows are global rows gathered from global_pos.
 * entries: 4 int32 per entry {src_row, flags, kb, lim}
 *          flags bits 0/1: query tile 0/1 computes this key tile,
 *          bits 2/3: the tile needs no predicate for query tile 0/1,
 *          bits 4-5: kind (0 band tile of the natural grid, 1 packed sparse
 *          columns [src_row, lim) of C, 2 dense causal walk for global rows).
 * which = 3: the key-major schedule of spattn_bwd's dK/dV pass.  Its "items" are
 *          64-key units {key0, entry_offset, entry_count, flags}; flags bit 0: the
 *          unit is packed sparse columns C[key0 .. key0+63] (these come first),
 *          else natural keys key0 .. key0+63.  Its entries are 64-row query groups
 *          {q0, flags, a, b}: flags bits 4-5 kind as above, bit 0: q0 indexes
 *          global_pos (rows gathered from the global list); bit 1: the local
 *          window alone allows every pair of the group's rows and the unit's keys
 *          (band entries only); a packed entry reads packed columns [a, b) of its
 *          unit.  Rows that are global tokens take part only in gathered entries.
 * which = 4: the same at 128-key units and 128-row groups: the schedule of the
 *          bf16 (tensor-core) dK/dV kernel.  Entry kind 3 (both key-major forms and
 *          the forward forms) is a key tile outside the band that only BigBird random
 *          blocks reach.
 * *n_items / *n_entries receive the sizes; arrays shorter than that are an
 * error (SPATTN_ERR_SHAPE) and nothing is written.  items/entries may be NULL to
 * query the sizes.  *tile_products receives the number of (query tile, key tile)
 * products one (batch, head) computes (which = 3: the number of entries).
 */
spattn_status spattn_plan_copy_schedule(const spattn_plan* plan, int32_t which, int32_t* items,
                                        int64_t item_cap, int64_t* n_items, int32_t* entries,
                                        int64_t entry_cap, int64_t* n_entries,
                                        int64_t* tile_products);

/* Enable (1) or disable (0) the device walk counter: every (query tile, key tile)
 * product the forward kernels compute adds one to a device counter, read with
 * spattn_plan_walk_count (synchronises the device).  Enabling resets it to 0. */
spattn_status spattn_plan_set_walk_counter(spattn_plan* plan, int32_t enable);
spattn_status spattn_plan_walk_count(const spattn_plan* plan, int64_t* count);

/*
 * Forward pass on device buffers, asynchronous on `cuda_stream`.
 * Q, K, V: [B, H, T, d] of `dtype` (bf16 or fp32), O: same shape and dtype,
 * LSE: [B, H, T] fp32 natural log (may be NULL to skip it).  scale > 0 and finite
 * (the glossary's 1/sqrt(d_k) is the usual choice).  bf16 runs on the tcgen05
 * tensor-core kernel (fp32 accumulation, fp32 online softmax); fp32 runs on FP32
 * FMA units.  The first call for a given B*H may allocate the plan's packing
 * scratch (cudaMalloc); later calls with the same or smaller B*H allocate
 * nothing.  Device-side waits are bounded: a wait that runs out sets a device
 * error word which the next spattn_fwd or spattn_plan_check_device call reports
 * as SPATTN_ERR_TIMEOUT.  Errors: NULL, SHAPE, DTYPE, ALIGN, INVALID_SPEC
 * (scale), CUDA, TIMEOUT.
 */
spattn_status spattn_fwd(const spattn_plan* plan, int32_t B, int32_t H, spattn_dtype dtype,
                         const void* Q, const void* K, const void* V, float scale, void* O,
                         float* LSE, void* cuda_stream);

/*
 * Backward pass (gradients) on device buffers, asynchronous on `cuda_stream`.
 * Given the forward's inputs Q, K, V, its output O and log-sum-exp LSE (as written
 * by spattn_fwd with the same plan, dtype and scale) and the gradient dO of a loss
 * with respect to O, writes dQ, dK, dV: the chain rule through the softmax over the
 * allowed set S_i ("Sparse attention" glossary, section "Choose the available
 * reads", differentiated):
 *   alpha_ij = exp(scale q_i.k_j - LSE_i),  D_i = dO_i . O_i,
 *   ds_ij = alpha_ij (dO_i . v_j - D_i)  for j in S_i (0 elsewhere),
 *   dQ_i = scale sum_j ds_ij k_j,  dK_j = scale sum_i ds_ij q_i,  dV_j = sum_i alpha_ij dO_i.
 * Q, K, V, O, dO, dQ, dK, dV: [B, H, T, d] of `dtype`, contiguous, 16-byte aligned;
 * LSE: [B, H, T] fp32 (required).  dQ, dK, dV are overwritten (every row is
 * written; nothing needs zeroing).  bf16 runs on the tcgen05 tensor cores (bf16
 * products, fp32 accumulation; P and dS rounded to bf16 as product operands), fp32
 * on FP32 FMA units; neither uses atomics (every row's dQ and every key's dK, dV is
 * summed inside one CTA), so the result is the same on every call.  Outputs of bf16
 * calls are rounded once, to nearest even.  The first call for a given B*H may
 * allocate the plan's backward scratch (row dots, packed-column partial sums and,
 * for bf16, packed copies of the sparse-column K, V and global-row Q, dO).
 * Errors: NULL, SHAPE, DTYPE, ALIGN, INVALID_SPEC (scale), CUDA.
 */
spattn_status spattn_bwd(const spattn_plan* plan, int32_t B, int32_t H, spattn_dtype dtype,
                         const void* Q, const void* K, const void* V, const void* O,
                         const float* LSE, const void* dO, float scale, void* dQ, void* dK,
                         void* dV, void* cuda_stream);

/*
 * ---- Decode: one generation step against a capped ring-buffer KV cache ----------
 *
 * The token at position t reads the w most recent positions max(0, t-w+1) .. t,
 * itself included ("Sparse and sliding-window attention", section "Sliding window
 * attention"); a sliding-window layer therefore keeps only the last cap >= w keys
 * and values ("Attention variants", section 1), whatever the length of the
 * generation.  Position p lives in slot p % cap of the cache.
 *
 * Layouts (device memory, contiguous, 16-byte aligned):
 *   K_cache, V_cache: [B, Hkv, cap, d] of `dtype` (caller-owned; slots outside the
 *                     window never affect the result, whatever they hold: bf16 reads
 *                     whole 64-slot blocks and masks the slots past the window);
 *   q, out:           [B, Hq, d] of `dtype`; lse: [B, Hq] fp32 natural log (or NULL);
 *   k_new, v_new:     [B, Hkv, d] of `dtype`;
 *   pos:              [B] int64, device memory: the position of the token each batch
 *                     row is generating (rows may be at different positions).  A
 *                     negative position means "no token": append skips the row and
 *                     decode writes out = 0, lse = -inf.
 * Query head h reads key/value head h / (Hq / Hkv) (grouped-query attention); Hq / Hkv
 * must be 1, 2, 4 or 8.  head_dim 64 or 128; 1 <= cap <= 2^30.
 */

/* Write k_new, v_new of every (b, kv head) to slot pos[b] % cap.  Asynchronous on
 * cuda_stream.  Errors: NULL, ALIGN, SHAPE, DTYPE, CUDA. */
spattn_status spattn_kv_append(int32_t B, int32_t Hkv, int64_t cap, int32_t head_dim,
                               spattn_dtype dtype, void* K_cache, void* V_cache,
                               const void* k_new, const void* v_new, const int64_t* pos,
                               void* cuda_stream);

/* Bytes of device workspace spattn_decode needs for these sizes (caller-owned).  The
 * first 4 bytes are the device error word: zero the workspace once (cudaMemset)
 * before its first use; spattn_decode_check reads and clears the word. */
spattn_status spattn_decode_workspace_bytes(int32_t B, int32_t Hq, int32_t Hkv, int64_t cap,
                                            int32_t head_dim, size_t* bytes);

/* One decode step: out[b, h] = sum over the allowed positions p of
 * softmax_p(scale q[b,h] . k_p) v_p with k_p, v_p read from slot p % cap of key/value
 * head h / (Hq/Hkv), the allowed positions being max(0, pos[b]-window+1) .. pos[b]
 * (window = 0 means window = cap; 1 <= window <= cap).  The caller appends the
 * step's own key and value (spattn_kv_append) before calling, as the token reads
 * itself.  Asynchronous on cuda_stream; fp32 accumulation.  bf16: products on the
 * tensor cores with the softmax weights rounded to bf16 for the weighted sum (as the
 * forward pass), out rounded once; fp32: FP32 products throughout.
 * Device-side waits are bounded: one that runs out sets the workspace's error word
 * (reported by spattn_decode_check as SPATTN_ERR_TIMEOUT).
 * Errors: NULL, ALIGN, SHAPE (also a workspace smaller than
 * spattn_decode_workspace_bytes), INVALID_SPEC (window, scale), DTYPE, CUDA. */
spattn_status spattn_decode(int32_t B, int32_t Hq, int32_t Hkv, int64_t cap, int64_t window,
                            int32_t head_dim, spattn_dtype dtype, const void* q,
                            const void* K_cache, const void* V_cache, const int64_t* pos,
                            float scale, void* out, float* lse, void* workspace,
                            size_t workspace_bytes, void* cuda_stream);

/* spattn_kv_append followed by spattn_decode, as one step: k_new, v_new ([B][Hkv]
 * [head_dim], 16-byte aligned, the dtype of the cache) are written to slot pos[b] % cap
 * and the step's query reads them, as the token reads itself ("Sparse and
 * sliding-window attention", section "Sliding window attention": position t reads
 * t - W + 1 .. t, with the cache capped at W).  For bf16 the decode kernel does the
 * append (the CTA that reads slot pos[b] % cap writes the rows to the cache and uses
 * them directly), so a step is two launches (decode, merge) instead of three; the
 * results are identical to the two calls.  For fp32 it launches the append kernel
 * first.  Same arguments, layouts, workspace and errors as spattn_decode, plus NULL /
 * ALIGN for k_new and v_new. */
spattn_status spattn_decode_append(int32_t B, int32_t Hq, int32_t Hkv, int64_t cap,
                                   int64_t window, int32_t head_dim, spattn_dtype dtype,
                                   const void* q, void* K_cache, void* V_cache,
                                   const void* k_new, const void* v_new, const int64_t* pos,
                                   float scale, void* out, float* lse, void* workspace,
                                   size_t workspace_bytes, void* cuda_stream);

/* Synchronise cuda_stream, then report (and clear) the decode workspace's error word:
 * SPATTN_ERR_TIMEOUT if a device-side wait ran out, else SPATTN_OK. */
spattn_status spattn_decode_check(void* workspace, void* cuda_stream);

/*
 * The same forward pass from HOST buffers: copies Q/K/V host -> device, runs
 * spattn_fwd, copies O and LSE device -> host, and returns once everything has
 * completed.  The (batch, head) units are processed in up to 16 chunks of consecutive
 * units as a pipeline: the host -> device copy of chunk k+1 (on a copy stream the
 * plan owns), the forward of chunk k (on `cuda_stream`) and the device -> host copy of
 * chunk k-1 (a second plan-owned stream) run at the same time; the copies start after
 * the work already queued on `cuda_stream`.  Results are identical to one spattn_fwd.
 * Host buffers should be pinned, or the copies neither reach full bandwidth nor
 * overlap.  The caller provides the device buffers (same shapes) so that this call
 * allocates nothing beyond spattn_fwd's scratch and, on first use, the plan's two
 * streams and their events.  LSE pointers may both be NULL.  Not safe to call on one
 * plan from two host threads at once.
 */
spattn_status spattn_fwd_host(const spattn_plan* plan, int32_t B, int32_t H,
                              spattn_dtype dtype, const void* Q_host, const void* K_host,
                              const void* V_host, float scale, void* O_host, float* LSE_host,
                              void* Q_dev, void* K_dev, void* V_dev, void* O_dev,
                              float* LSE_dev, void* cuda_stream);

/*
 * The forward pass of spattn_fwd for callers that cannot allocate device memory
 * (a process whose GPU memory is owned by another allocator, or a loop that must
 * never pay for a cudaMalloc after start-up).  The method on the pages has no
 * counterpart: this is a memory-management variant only.  Same arguments, layouts,
 * results and errors as spattn_fwd, but the packing scratch (packed strided /
 * global key columns and gathered global query rows) comes from one fixed 16 MiB
 * array in the library's device memory, held by every GPU that loads the library
 * until the process exits, so the call allocates nothing.  The scratch needed is
 * B*H*(2*n_columns + n_global)*d*element_size bytes; above 16 MiB the call returns
 * SPATTN_ERR_SHAPE and launches nothing.  The first call on each device looks up
 * the array's device address (cudaGetSymbolAddress, with that device current) and
 * remembers it with the current CUDA context; a call made in a new context on that
 * device (after cudaDeviceReset, say) looks it up again.  Make the first call on a
 * device, and the first after any such reset, before any stream capture.  All calls share the array:
 * calls that may overlap on the GPU (unordered streams) race and give wrong results.
 */
spattn_status spattn_fwd_static_scratch(const spattn_plan* plan, int32_t B, int32_t H,
                                        spattn_dtype dtype, const void* Q, const void* K,
                                        const void* V, float scale, void* O, float* LSE,
                                        void* cuda_stream);

/* Time budget, in SM clock cycles, of every device-side wait of the bf16 forward
 * kernel (default 8e9, about 4 s at 2 GHz).  A wait that runs out records
 * SPATTN_ERR_TIMEOUT in the plan's device error word; the kernel then drains its
 * in-flight copies and products, frees its tensor memory and returns, so the CUDA
 * context stays usable.  Errors: NULL, SHAPE (cycles == 0). */
spattn_status spattn_plan_set_wait_budget(spattn_plan* plan, uint64_t cycles);

/* Test hook for the failure path above: while enabled, the bf16 forward kernel's
 * MMA warp first waits on a barrier that nothing signals, so that wait runs out of
 * its budget (set a short one first) and the call's error word reports
 * SPATTN_ERR_TIMEOUT through spattn_plan_check_device.  No fault, trap or unbounded
 * wait is involved.  The outputs of such a call are unspecified. */
spattn_status spattn_plan_test_wait_timeout(spattn_plan* plan, int32_t enable);

/* Synchronise `cuda_stream` and report (then clear) the plan's device error word:
 * SPATTN_OK, SPATTN_ERR_TIMEOUT or SPATTN_ERR_CUDA. */
spattn_status spattn_plan_check_device(const spattn_plan* plan, void* cuda_stream);

/* Free a plan and its device memory (NULL is a no-op).  Synchronises the device
 * first so no in-flight kernel still reads it. */
void spattn_plan_destroy(spattn_plan* plan);

/* Message for the last failing call on this thread ("" if none). */
const char* spattn_last_error(void);

/* Library version string. */
const char* spattn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SPATTN_H_ */
