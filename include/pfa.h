/*
 * pfa.h -- C ABI of the GB300 (sm_103a) chunked causal GQA prefill-attention
 * library (libpfa.so).
 *
 * The operation is one layer's self-attention for a chunk of T query tokens
 * at absolute positions start_pos .. start_pos+T-1 against a KV cache that
 * already holds L = start_pos + T positions, as defined on the gnosis page
 * "Prefill attention -> GPU: handoff", section "GPU design":
 *
 *   - GQA: group = num_heads / num_kv_heads; query head h reads kv head
 *     h / group (integer division).
 *   - scores s_j = scale * <q[t][h][:], k[h/group][j][:]>, scaled before the
 *     row maximum and softmax (scale is usually 1/sqrt(head_dim)).
 *   - causal mask: key j is visible to token t only if j <= start_pos + t
 *     (masked scores contribute exactly zero weight).
 *   - sliding window (the "causal(+windowed)" per-row [lo, hi] band of the
 *     TensorSharp2 Gemma-4 prefill design, section 5 Option A): when
 *     window > 0, key j is also required to satisfy j > start_pos + t - window,
 *     so a row sees min(pos + 1, window) keys, its own position included.
 *   - out[t][h][:] = sum_j softmax(s)_j * v[h/group][j][:].
 *
 * Every row has at least one visible key (its own position), so no row is
 * ever empty.
 */
#ifndef PFA_H
#define PFA_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PFA_API __attribute__((visibility("default")))
#else
#define PFA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Element type of q, k_cache, v_cache and out (all four share it). */
typedef enum {
    PFA_F32 = 0,   /* fp32 in, fp32 out, fp32 arithmetic throughout          */
    PFA_BF16 = 1   /* bf16 in, bf16 out (round-to-nearest-even), fp32 accumulation */
} pfa_dtype;

/* Status codes.  Every entry point returns one of these and never aborts,
 * traps or prints (unless the environment variable PFA_TRACE is set, which
 * makes the launch path print one line per call to stderr). */
typedef enum {
    PFA_OK = 0,
    PFA_ERR_NULL = -1,       /* a required pointer is NULL                          */
    PFA_ERR_SHAPE = -2,      /* T < 0, start_pos < 0, heads <= 0, H % Hkv != 0,
                                unsupported head_dim, or a size beyond the limits   */
    PFA_ERR_DTYPE = -3,      /* dtype is not a pfa_dtype value                      */
    PFA_ERR_ALIGNMENT = -4,  /* a pointer is not 16-byte aligned                    */
    PFA_ERR_DEVICE = -5,     /* no usable device, or not an sm_103 (GB300) device,
                                or a pointer that is not device-accessible memory   */
    PFA_ERR_LAUNCH = -6,     /* the CUDA runtime refused the launch                 */
    PFA_ERR_TIMEOUT = -7,    /* a device-side wait gave up (reported after a sync
                                by pfa_last_device_error)                           */
    PFA_ERR_VALUE = -8,      /* scale is not a finite number                        */
    PFA_ERR_ALIAS = -9,      /* out overlaps q, k_cache or v_cache                  */
    PFA_ERR_SCRATCH = -10,   /* the shape needs more scratch than
                                pfa_prefill_attention_noalloc holds                 */
    PFA_ERR_LENGTHS = -11    /* pfa_prefill_attention_graph: the {T, start_pos} read
                                on the device did not fit its capacities (reported
                                after a sync by pfa_last_device_error)              */
} pfa_status;

/*
 * pfa_prefill_attention -- asynchronous prefill attention on `stream`.
 *
 *   q        device pointer, [T][num_heads][head_dim] contiguous, dtype.
 *            Token-major, as the page's batch_q rows (section "GPU design",
 *            "Layout").
 *   k_cache  device pointer, [num_kv_heads][L][head_dim] contiguous, dtype,
 *            L = start_pos + T: each kv head's keys form one contiguous
 *            [L x head_dim] block (the page's kv_cache.keys layout with
 *            capacity L).  Positions start_pos .. L-1 must already hold the
 *            chunk's own keys.
 *   v_cache  device pointer, same layout as k_cache.
 *   out      device pointer, [T][num_heads][head_dim] contiguous, dtype.  It
 *            must not overlap q, k_cache or v_cache.  Every element is
 *            written.
 *   T        number of query tokens in the chunk (T == 0 is a no-op).
 *   start_pos  absolute position of the chunk's first token (>= 0).
 *   num_heads, num_kv_heads  query and kv head counts; num_heads must be a
 *            multiple of num_kv_heads.  For PFA_BF16 the group size
 *            num_heads / num_kv_heads must be at most 128.
 *   head_dim 128 or 512 for PFA_BF16; any multiple of 4 up to 512 for PFA_F32.
 *   window   <= 0: global causal attention; > 0: sliding window of that many
 *            keys (key j visible iff start_pos+t-window < j <= start_pos+t).
 *   scale    multiplier of the dot products, applied as given (finite).
 *   dtype    a pfa_dtype value.
 *   stream   cudaStream_t to launch on; NULL means the legacy default stream.
 *
 * Ownership: the caller owns all four buffers and keeps them alive until the
 * work on `stream` completes.  The library allocates no device memory for
 * this call; it caches TMA tensor-map descriptors (host memory) keyed by
 * pointer and shape, and per-device launch attributes.  It launches one
 * kernel per call (one query-tile pair per CTA); see pfa_prefill_attention_ws
 * for the balanced schedule.
 *
 * Behaviour: validates the arguments, then enqueues the kernel(s) on `stream`
 * and returns without synchronising.  Validation failures return a status
 * before anything is enqueued.  A device-side wait that exceeds its time
 * limit makes the kernel record PFA_ERR_TIMEOUT and return early; read it
 * with pfa_last_device_error.  The result is a deterministic function of the
 * inputs: repeated calls produce bit-identical outputs.
 *
 * Returns PFA_OK or a pfa_status error code.
 */
PFA_API int pfa_prefill_attention(const void *q, const void *k_cache, const void *v_cache, void *out,
                          int64_t T, int64_t start_pos, int num_heads, int num_kv_heads,
                          int head_dim, int window, float scale, int dtype, void *stream);

/*
 * pfa_prefill_attention_ws -- pfa_prefill_attention with a caller-provided
 * device workspace that enables the split-key schedules.
 *
 *   workspace        device pointer (256-byte aligned) or NULL, not
 *                    overlapping q, k_cache, v_cache or out.  Its contents on
 *                    entry do not matter; the call may overwrite all of it.
 *   workspace_bytes  its size.  If it is smaller than the value
 *                    pfa_workspace_bytes reports for the same shape (or the
 *                    workspace is NULL), the call uses the plain schedule,
 *                    exactly as pfa_prefill_attention does.
 *
 * The balanced schedule (head_dim 128, bf16, caches small enough to stay in
 * L2) cuts the key-tile work of all query tiles into one equal share per SM
 * instead of one CTA per query-tile pair; query tiles whose keys are split
 * between SMs leave fp32 partial results (output, exponent base, row sum) in
 * the workspace, which a second kernel on the same stream combines in a fixed
 * order.  The result is deterministic for a given device and shape, and equal
 * to the plain schedule's within floating-point reassociation (both are
 * within the stated tolerance of the exact result).  For bf16 with head_dim
 * 512 the workspace enables the tail split only (see pfa_schedule): the
 * whole waves of query tiles run whole, and each tile of a last, partial
 * wave is cut into equal key ranges whose partial results are combined in
 * key order.  Concurrent calls must
 * not share a workspace.  Other arguments, ownership and errors: as for
 * pfa_prefill_attention (PFA_ERR_ALIGNMENT / PFA_ERR_DEVICE / PFA_ERR_ALIAS
 * also cover the workspace).
 */
PFA_API int pfa_prefill_attention_ws(const void *q, const void *k_cache, const void *v_cache,
                                     void *out, int64_t T, int64_t start_pos, int num_heads,
                                     int num_kv_heads, int head_dim, int window, float scale,
                                     int dtype, void *workspace, size_t workspace_bytes,
                                     void *stream);

/*
 * pfa_prefill_attention_cache -- pfa_prefill_attention_ws on the caller's own
 * buffer layout instead of the contiguous one.  The layouts are those of the
 * gnosis page "Prefill attention -> GPU: handoff" (section "GPU design",
 * "Layout": Q rows of qkv_dim elements in batch_q, kv head kh's block at
 * kh * max_seq_len * head_dim, the output scattered back into rows of
 * qkv_dim) and the circular cache of sliding-window layers in the
 * TensorSharp2 Gemma-4 prefill design (section 4, R4: position pos is stored
 * at index pos % capacity).
 *
 *   q        element (t, h, d) at q[t * qkv_dim + h * head_dim + d].
 *   out      element (t, h, d) at out[t * qkv_dim + h * head_dim + d]; only
 *            these T * num_heads * head_dim elements are written, the rest of
 *            each row is left as it was.  out must not overlap q, k_cache or
 *            v_cache (taken as their full spans).
 *   k_cache, v_cache
 *            key j of kv head kh at k_cache[kh * max_seq_len * head_dim +
 *            row(j) * head_dim + d], row(j) = j (ring == 0) or
 *            j % max_seq_len (ring != 0).
 *   qkv_dim  elements from one token's row to the next in q and out;
 *            >= num_heads * head_dim, and qkv_dim * element size must be a
 *            multiple of 16 bytes (PFA_ERR_ALIGNMENT otherwise).
 *   max_seq_len  rows allocated per kv head (> 0).  With ring == 0 it must be
 *            >= L = start_pos + T (rows past L are never read).
 *   ring     non-zero: circular cache.  Needs window > 0 and
 *            max_seq_len >= min(L, window + T - 1), so that every key a row of
 *            the chunk sees is still stored (the caller has written positions
 *            start_pos .. L-1 at row(j), overwriting the oldest).  For PFA_BF16,
 *            once the ring has wrapped (L > max_seq_len) max_seq_len must be a
 *            multiple of 128, the key-tile height.
 *   workspace, workspace_bytes  as for pfa_prefill_attention_ws.
 *
 * With qkv_dim = num_heads * head_dim, max_seq_len = L and ring = 0 it is
 * exactly pfa_prefill_attention_ws.  Layout errors return PFA_ERR_SHAPE
 * (or PFA_ERR_ALIGNMENT) before anything is enqueued.  Ownership, behaviour,
 * other errors and determinism: as for pfa_prefill_attention_ws.
 */
PFA_API int pfa_prefill_attention_cache(const void *q, const void *k_cache, const void *v_cache,
                                        void *out, int64_t T, int64_t start_pos, int num_heads,
                                        int num_kv_heads, int head_dim, int window, float scale,
                                        int dtype, int64_t qkv_dim, int64_t max_seq_len, int ring,
                                        void *workspace, size_t workspace_bytes, void *stream);

/*
 * pfa_workspace_bytes -- bytes of workspace the balanced schedule needs for
 * this shape on the current device (0 when it would not be used).  Same
 * shape validation as pfa_prefill_attention; no pointers are needed and
 * nothing is launched.  Returns PFA_OK and sets *bytes, or an error status.
 */
PFA_API int pfa_workspace_bytes(int64_t T, int64_t start_pos, int num_heads, int num_kv_heads,
                                int head_dim, int window, int dtype, size_t *bytes);

/*
 * pfa_prefill_attention_graph -- pfa_prefill_attention_cache with the chunk's
 * length and position read from device memory when the kernel runs, so that
 * one captured CUDA graph replays for any chunk: the launch's parameters and
 * grid depend only on capacities.  This is the graph-replay requirement of
 * the TensorSharp2 Gemma-4 prefill design (section 4, R5: inputs refreshed
 * in place, the same pointers and shapes every chunk; section 6, Phase 2) and
 * of the FreeToken draft-graph change ("replay holds at any sequence length":
 * the lengths live in fixed device buffers written before each replay).
 *
 *   lengths  device pointer (8-byte aligned) to two int64: {T, start_pos} of
 *            the chunk, read by the kernel at run time (write them on the
 *            stream, or before it, ahead of each launch or replay).
 *   max_T    the largest T: q and out hold max_T rows of qkv_dim elements;
 *            the grid is sized for it (CTAs beyond the run-time chunk exit at
 *            once).  1 <= max_T <= max_seq_len (max_T == 0 is a no-op).
 *   q, k_cache, v_cache, out, num_heads .. dtype, qkv_dim, max_seq_len, ring
 *            as for pfa_prefill_attention_cache; for PFA_BF16 a ring's
 *            max_seq_len must be a multiple of 128.
 *
 * Run-time checks: 0 <= T <= max_T, start_pos >= 0, and L = start_pos + T <=
 * max_seq_len (linear) or max_seq_len >= min(L, window + T - 1) (ring).  A
 * launch whose lengths fail them writes nothing and records PFA_ERR_LENGTHS,
 * which pfa_last_device_error returns.  T == 0 writes nothing.
 *
 * Cache rows past L: the host cannot clip the tensor maps at a run-time L, so
 * for PFA_BF16 the rows of the last 128-key tile past L are read and
 * weighted by exactly zero -- they must hold finite values
 * (never-written rows of a zero-initialised cache do).  The fp32 path reads
 * no row past L.
 *
 * Always the plain schedule (no workspace).  Capture: the first call of the
 * library on a device does per-device set-up (device queries, a memset of
 * the device error word, kernel attributes) that must not happen inside a
 * stream capture; make one call of any entry point on the device first.
 * Other behaviour, ownership and errors: as for pfa_prefill_attention_cache.
 */
PFA_API int pfa_prefill_attention_graph(const void *q, const void *k_cache, const void *v_cache,
                                        void *out, const int64_t *lengths, int64_t max_T,
                                        int num_heads, int num_kv_heads, int head_dim, int window,
                                        float scale, int dtype, int64_t qkv_dim,
                                        int64_t max_seq_len, int ring, void *stream);

/*
 * pfa_schedule -- which schedule pfa_prefill_attention_ws runs for this shape
 * on the current device when its workspace is at least *workspace_bytes
 * (the value pfa_workspace_bytes reports):
 *   PFA_SCHEDULE_PLAIN     one kernel, one CTA per pair of 128-row query tiles
 *                          (head_dim 512: per pair of query tiles, two
 *                          clusters of two CTAs, one cluster per half of the
 *                          output columns);
 *   PFA_SCHEDULE_BALANCED  equal-cost runs of key-tile ranges per SM, then a
 *                          merge kernel (two launches);
 *   PFA_SCHEDULE_TAIL      the whole waves of pairs run whole and the pairs
 *                          of the last, partial wave are cut into equal key
 *                          ranges (with no more pairs than SMs: every pair
 *                          is cut, the CTAs of one range running together),
 *                          then a merge kernel (two launches).  head_dim 512
 *                          has this schedule (without the every-pair form)
 *                          and the plain one; fp32 has the plain one only.
 * Same validation as pfa_workspace_bytes; nothing is launched.  Returns
 * PFA_OK and sets both outputs, or an error status.
 */
#define PFA_SCHEDULE_PLAIN 0
#define PFA_SCHEDULE_BALANCED 1
#define PFA_SCHEDULE_TAIL 2
PFA_API int pfa_schedule(int64_t T, int64_t start_pos, int num_heads, int num_kv_heads,
                         int head_dim, int window, int dtype, int *schedule,
                         size_t *workspace_bytes);

/*
 * pfa_host_buffer_bytes -- bytes of device memory pfa_prefill_attention_host
 * needs for this shape on the current device: the device copies of q,
 * k_cache, v_cache and out, then one workspace per group of kv heads (bf16:
 * the size pfa_workspace_bytes gives for the group's heads alone), each
 * rounded up to 256 bytes.  Same validation as
 * pfa_workspace_bytes; nothing is launched.  Returns PFA_OK and sets *bytes
 * (0 for T == 0), or an error status.
 */
PFA_API int pfa_host_buffer_bytes(int64_t T, int64_t start_pos, int num_heads, int num_kv_heads,
                                  int head_dim, int window, int dtype, size_t *bytes);

/*
 * pfa_prefill_attention_host -- the operation of pfa_prefill_attention on
 * HOST buffers: the batch buffers of the gnosis page "Prefill attention ->
 * GPU: handoff" (section "GPU design", "Layout": q rows and the kv cache
 * already populated on the host), copied to the device once per call into
 * one caller-owned device buffer (section "Implementation status", open
 * item 3: pool the device buffers instead of per-tile copies and
 * allocations), with the copies overlapped with the attention kernels (the
 * same page's "Expected ceiling" counts the per-layer host-device copies in
 * the GPU time).
 *
 *   q, k_cache, v_cache  host, read only; the layouts of
 *                        pfa_prefill_attention ([T][H][D], [Hkv][L][D]).
 *   out                  host, [T][H][D]; written by a device-to-host copy
 *                        that completes with the stream's work.
 *   device_buffer        device memory on the current device, 256-byte
 *                        aligned, of at least pfa_host_buffer_bytes(...)
 *                        bytes (caller-owned; the call stores the device
 *                        copies there).  Must not be in use by other work
 *                        that can run at the same time.
 *   device_buffer_bytes  its size.
 *   other arguments      as for pfa_prefill_attention.
 *
 * Host buffers should be page-locked (cudaHostAlloc / cudaHostRegister) for
 * the copies to be asynchronous and at full speed; pageable memory works,
 * with copies the driver stages (partly synchronous to the host).
 *
 * Behaviour: asynchronous on `stream`; nothing is allocated.  The kv heads
 * are processed in up to four groups (one when the call moves less than
 * 4 MiB, two below 128 MiB, else four): each group's K/V rows and q columns
 * are copied in (groups in order, so the first group's kernel starts while
 * the later groups' data is still on its way), its kernel runs on its own
 * copy of the group (with the schedule pfa_prefill_attention_ws picks for
 * the group's heads, in the group's workspace), and its
 * out columns are copied back while later groups compute.  The groups run
 * on streams of the library's own (created on the first call on a device,
 * kept until the process exits) that wait for the work queued on `stream`
 * before the call and that `stream` waits for in turn: synchronise `stream`
 * (or wait for an event recorded on it after the call) before reading out.
 * Each head's result is the one pfa_prefill_attention_ws computes for the
 * group's heads alone: bit-identical to pfa_prefill_attention where the group
 * runs the plain schedule, else equal within the split schedules' merge.
 *
 * Errors: PFA_ERR_NULL for a null pointer, PFA_ERR_ALIGNMENT for a device
 * buffer that is not 256-byte aligned or host buffers that are not 16-byte
 * aligned, PFA_ERR_SHAPE for a device buffer smaller than required or the
 * shape errors of pfa_prefill_attention, PFA_ERR_DEVICE when the device
 * buffer is not device memory of the current device, PFA_ERR_LAUNCH when a
 * copy or a launch is refused.  Nothing is enqueued on an argument error.
 */
PFA_API int pfa_prefill_attention_host(const void *q, const void *k_cache, const void *v_cache,
                                       void *out, int64_t T, int64_t start_pos, int num_heads,
                                       int num_kv_heads, int head_dim, int window, float scale,
                                       int dtype, void *device_buffer, size_t device_buffer_bytes,
                                       void *stream);

/*
 * pfa_prefill_attention_noalloc -- the call of pfa_prefill_attention_ws with
 * the balanced schedule, for callers that cannot allocate device memory.
 * (The source pages have no counterpart: this is an interface convenience.)
 *
 * Who needs it: a caller that must not or cannot call cudaMalloc around the
 * call -- code being captured into a CUDA graph, code under an allocator that
 * owns all device memory, a host integration with no device allocator -- and
 * so cannot hand pfa_prefill_attention_ws a workspace.  This entry point uses
 * scratch memory that belongs to the library instead: a static array of
 * PFA_NOALLOC_SCRATCH_BYTES (32 MiB) in device memory, present on every
 * device where the library's code has been loaded, until the process exits.
 * It allocates nothing: no cudaMalloc/cudaFree and no allocating library
 * routine is called.
 *
 * Arguments, layouts, ownership and the result: as for pfa_prefill_attention.
 * For bf16 with head_dim 128 it runs the schedule pfa_schedule reports (the
 * balanced or the tail-split one) in the static scratch; a shape whose
 * schedule needs more than PFA_NOALLOC_SCRATCH_BYTES is refused with
 * PFA_ERR_SCRATCH before anything is launched (long chunks deep in a
 * context, whose tail split needs ~92 MiB for a 2048-token chunk of 32
 * heads, are refused; pfa_prefill_attention runs them with the plain
 * schedule).  It refuses rather than quietly running the plain schedule so
 * that one promise holds: whenever it returns PFA_OK, its output is
 * bit-identical to that of pfa_prefill_attention_ws given a large enough
 * workspace.  Shapes that use no workspace (other dtypes or head_dims, or
 * shapes where the plain schedule is picked) run as pfa_prefill_attention.
 *
 * Sharing: every call on a device uses the same scratch and leaves its own
 * partial results in it.  No part of it needs to be zero on entry (a call
 * only reads what it wrote itself).  Calls whose kernels may overlap on the
 * GPU -- on different streams without an ordering between them -- race on
 * the scratch and can return wrong results; order them.
 *
 * Set-up: the first call on a device looks up the scratch's device address
 * (cudaGetSymbolAddress, with that device current).  Make that first call
 * before any stream capture that includes this entry point.
 */
#define PFA_NOALLOC_SCRATCH_BYTES (32u << 20)
PFA_API int pfa_prefill_attention_noalloc(const void *q, const void *k_cache,
                                          const void *v_cache, void *out, int64_t T,
                                          int64_t start_pos, int num_heads, int num_kv_heads,
                                          int head_dim, int window, float scale, int dtype,
                                          void *stream);

/* Human-readable name of a pfa_status value (static storage, never NULL). */
PFA_API const char *pfa_status_string(int status);

/*
 * pfa_last_device_error -- synchronise `stream`, then return and clear the
 * device-side error word of the current device: PFA_OK, PFA_ERR_TIMEOUT if
 * a kernel launched since the last call gave up on a wait, or
 * PFA_ERR_LENGTHS if a pfa_prefill_attention_graph launch found its
 * run-time lengths out of range (timeouts take precedence).  Returns
 * PFA_ERR_DEVICE if the stream cannot be synchronised (the CUDA error is then
 * the runtime's).
 */
PFA_API int pfa_last_device_error(void *stream);

/*
 * pfa_debug_check_schedule -- test hook, host only (no device is touched):
 * replays, for the bf16 head_dim-128 path of this shape on a GPU with
 * `num_sms` SMs, the work assignment the kernels would execute with a large
 * enough workspace -- every CTA's (query-tile pair, key-tile range, partial
 * slot) items and the merge entries -- and checks its invariants: each key
 * tile of each pair is computed exactly once, key tiles lie inside the cache
 * and hold a visible key, whole-pair items write the output and partial items
 * own distinct workspace slots that fit the workspace, and the merge combines
 * exactly the split pairs' pieces in key order.
 *   schedule      out: PFA_SCHEDULE_* of the shape
 *   ctas          out: CTAs of the main kernel
 *   failed_check  out: 0 when every invariant holds, else the number of the
 *                 first failed check
 * Returns PFA_OK (with the outputs set), PFA_ERR_NULL or PFA_ERR_SHAPE.
 */
PFA_API int pfa_debug_check_schedule(int64_t T, int64_t start_pos, int num_heads,
                                     int num_kv_heads, int window, int num_sms, int *schedule,
                                     int *ctas, int *failed_check);

/*
 * pfa_debug_check_schedule_d512 -- test hook, host only (no device is
 * touched): the same replay for the bf16 head_dim-512 path -- every CTA of the
 * grid mapped to its cluster, rank (query tile of the pair), output half and
 * key-tile range, and the merge's reads -- with its invariants: every output
 * half of every query tile is written by exactly one whole item or merged from
 * pieces that cover its pair's key tiles in order from distinct workspace
 * slots (each filled by the pair's two CTAs for both halves) that fit the
 * workspace; every cluster walks at least one key tile, its key tiles start
 * inside the cache and cover every key visible to its rows; the TMA boxes'
 * column coordinates are 16-byte aligned and inside the head; a query tile
 * past T occurs only as the second tile of an odd last pair.
 * Outputs and return values as for pfa_debug_check_schedule.
 */
PFA_API int pfa_debug_check_schedule_d512(int64_t T, int64_t start_pos, int num_heads,
                                          int num_kv_heads, int window, int num_sms,
                                          int *schedule, int *ctas, int *failed_check);

/* Library ABI version: (major << 16) | minor. */
PFA_API int pfa_version(void);

/*
 * pfa_debug_configure -- test hook for the device-side wait limits.
 *   wait_limit_ms  time limit of every device-side wait in later launches
 *                  (<= 0 restores the default of 2000 ms).
 *   force_timeout  non-zero makes the next tensor-core launches (bf16, and
 *                  fp32 with head_dim 128) wait once on a barrier that
 *                  nothing signals, so the limit expires and the
 *                  kernel takes its early-exit path (PFA_ERR_TIMEOUT);
 *                  zero restores normal operation.
 * Process-wide setting; not thread-safe with concurrent launches.
 * Returns PFA_OK.
 */
PFA_API int pfa_debug_configure(double wait_limit_ms, int force_timeout);

#ifdef __cplusplus
}
#endif

#endif /* PFA_H */
