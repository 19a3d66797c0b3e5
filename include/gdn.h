/*
 * gdn.h -- C ABI of the GB300 (sm_103a) gated delta rule library, libgdn.so.
 *
 * The operation (ferrox-core `gdn_chunk.rs`, module docs, "The algebra";
 * metaltile-std `gated_delta_wy.rs`, module docs, "Algorithm"): for every
 * batch b and value head hv a state S (Dv x Dk, fp32) is carried through the
 * tokens t of a sequence as
 *
 *     d_t = beta_t (v_t - g_t S_{t-1} k_t)
 *     S_t = g_t S_{t-1} + d_t k_t^T
 *     y_t = S_t q_t / sqrt(Dk)
 *
 * where g_t in (0, 1] is a multiplicative decay, beta_t the write strength,
 * and q_t, k_t are read from key head hk = hv / (Hv / Hk) (grouped GQA map,
 * metaltile-std `gated_delta_wy.rs`, "Layouts").
 *
 * Layouts (row-major, contiguous, every pointer a DEVICE pointer):
 *     q, k        [B, T, Hk, Dk]     dtype
 *     v, y        [B, T, Hv, Dv]     dtype
 *     g, beta     [B, T, Hv]         dtype
 *     state_in    [B, Hv, Dv, Dk]    fp32 (always)
 *     state_out   [B, Hv, Dv, Dk]    fp32 (always)
 * (metaltile-std `gated_delta_wy.rs`, "Layouts"; the state stays fp32.)
 *
 * Ownership: the caller owns every buffer, including any workspace; the
 * library makes no device allocation at run time (the fixed scratch of
 * gdn_prefill_noalloc is a static array of the library image, in device
 * memory once the library's kernels are loaded into a CUDA context).
 * All work is enqueued on `stream` (a cudaStream_t; NULL means the legacy
 * default stream) and the calls return without synchronising.
 * state_in == state_out (in place) is allowed; any other overlap between
 * inputs and outputs is undefined.
 *
 * Errors: every argument is checked on the host before anything is
 * launched; on a non-zero return nothing has been enqueued and the outputs
 * are untouched (except GDN_ERR_CUDA, see below).  No exception crosses
 * the ABI.  gdn_status_string() names a code.
 */
#ifndef GDN_H_
#define GDN_H_

#include <stddef.h>

#if defined(__GNUC__)
#define GDN_API __attribute__((visibility("default")))
#else
#define GDN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
#define GDN_OK                  0
#define GDN_ERR_INVALID       (-1) /* NULL required pointer, a size <= 0, Hv % Hk != 0 */
#define GDN_ERR_UNSUPPORTED   (-2) /* Dk/Dv not 64/128/256, chunk not 16/32/64, bad dtype,
                                      or a size beyond the limits: B*Hv > 2^20,
                                      B*T > 2^31 - 1, B*Hv*ceil(T/16) > 2^24 */
#define GDN_ERR_ALIGNMENT     (-3) /* a pointer that is not 16-byte aligned */
#define GDN_ERR_WORKSPACE     (-4) /* workspace NULL or smaller than gdn_prefill_workspace_bytes */
#define GDN_ERR_CUDA          (-5) /* the CUDA runtime reported an error at launch; the
                                      outputs are then unspecified */
#define GDN_ERR_DEVICE_TIMEOUT (-6) /* a kernel's bounded wait gave up (see gdn_device_status) */
#define GDN_ERR_NOALLOC_LIMIT (-7) /* gdn_prefill_noalloc: the problem needs more scratch than
                                      GDN_NOALLOC_SCRATCH_BYTES */

/* Element types of q, k, v, g, beta and y. */
#define GDN_DTYPE_F32   0
#define GDN_DTYPE_BF16  1
/* fp16: as bf16 (decode and T <= 32 on the row-packed kernels; longer
 * prefills with Dk = Dv = 128 on the tensor cores, in fp16 operands). */
#define GDN_DTYPE_F16   2

/*
 * Input conventions for gdn_prefill_ex / gdn_decode_step_ex (bits of
 * `options`; 0 gives gdn_prefill / gdn_decode_step exactly).
 *   GDN_OPT_TILED_HEADS  value head hv reads key head hv % Hk ("tiled"), instead
 *                        of hv / (Hv/Hk) ("grouped").  ferrox-core `gdn_chunk.rs`
 *                        names both maps (HeadMap::Tiled, HeadMap::Grouped) but
 *                        shows no body for either; these are the two usual GQA
 *                        layouts, the grouped one matching metaltile-std "Layouts".
 *   GDN_OPT_LOG_GATE     g holds log-decays (<= 0) and the decay is exp(g), as in
 *                        ferrox-core `delta_chunk` (`a = exp(g)`), instead of the
 *                        multiplicative gate of metaltile-std.
 *   GDN_OPT_L2NORM_QK    every q and k row (Dk values) is used as x / |x|,
 *                        computed in fp32 from the stored values (the step
 *                        before the recurrence in the MLX PR's test inputs); a
 *                        zero row stays zero.  For bf16 or fp16 inputs the
 *                        normalised rows enter the tensor-core products
 *                        rounded to the input type.
 * Any other bit gives GDN_ERR_UNSUPPORTED.
 */
#define GDN_OPT_TILED_HEADS 1
#define GDN_OPT_LOG_GATE    2
#define GDN_OPT_L2NORM_QK   4

/*
 * Bytes of device workspace gdn_prefill needs for this shape (0 if none).
 * Returns 0 as well for arguments gdn_prefill would reject.
 */
GDN_API size_t gdn_prefill_workspace_bytes(int B, int T, int Hk, int Hv, int Dk, int Dv,
                                   int chunk, int dtype);

/*
 * Prefill: run T tokens of every (b, hv) through the rule, chunk by chunk
 * (the chunked Woodbury-Young form of metaltile-std `gated_delta_wy.rs`,
 * "Algorithm" steps 1-9, with the decay ratios formed as products as in
 * ferrox-core `gdn_chunk.rs`, "The algebra").  Writes y for every token and
 * the state after token T-1 into state_out.
 *
 *   state_in   NULL means S_0 = 0.
 *   chunk      tokens per chunk: 16, 32 or 64.  Any T >= 1 is accepted; a
 *              last chunk shorter than `chunk` behaves as if padded with
 *              g = 1, beta = 0 tokens (metaltile-std kernel, chunk loop).
 *              Sequences of T <= 32 run a kernel of their own with the state
 *              on chip and no workspace (the short-T routing of the MLX PR
 *              "Pack gated_delta_seq", Performance): for bf16 / fp16 inputs
 *              with Dk = Dv = 128 the sequence as one chunk on warp-level
 *              tensor-core MMAs, otherwise the sequential rule in fp32.
 *   workspace  device scratch of at least gdn_prefill_workspace_bytes(...)
 *              bytes, 256-byte aligned, owned by the caller; its contents on
 *              entry do not matter and on return are unspecified.  It must
 *              not be used by anything else until the work on `stream` is done.
 *   stream     cudaStream_t, or NULL.
 * Dk and Dv are each 64, 128 or 256.  bf16 and fp16 inputs with Dk = Dv = 128,
 * 64 or 256 run on the tensor cores (tcgen05 at 128, warp-level MMAs in
 * chunks of 32 at 64 and 256), whose operands (the inputs and the per-chunk
 * intermediates) are then rounded to the input type and whose products
 * accumulate in fp32; every other head pair and fp32 inputs run the fp32
 * chunked path, which for Dk = Dv = 256 runs a chunk of 64 as two chunks of
 * 32.  The chunk size changes the result only by rounding, and
 * gdn_prefill_workspace_bytes accounts for the one each path uses.  Returns
 * GDN_OK or a GDN_ERR_* code.
 */
GDN_API int gdn_prefill(const void *q, const void *k, const void *v, const void *g,
                const void *beta, const float *state_in, float *state_out, void *y,
                int B, int T, int Hk, int Hv, int Dk, int Dv, int chunk,
                int dtype, void *workspace, size_t workspace_bytes, void *stream);

/* gdn_prefill with input conventions `options` (GDN_OPT_* bits above). */
GDN_API int gdn_prefill_ex(const void *q, const void *k, const void *v, const void *g,
                const void *beta, const float *state_in, float *state_out, void *y,
                int B, int T, int Hk, int Hv, int Dk, int Dv, int chunk,
                int dtype, void *workspace, size_t workspace_bytes, void *stream,
                int options);

/*
 * Decode: one token (T = 1) of every (b, hv) through the rule, streaming
 * the state once (the single-step recurrence above; row packing after the
 * MLX `gated_delta_seq` packed layout, PR "Pack gated_delta_seq: 8 value
 * rows per SIMD-group").
 *
 *   q, k [B, 1, Hk, Dk]; v, y [B, 1, Hv, Dv]; g, beta [B, 1, Hv]
 *   state_in must not be NULL; state_out may equal state_in (in place).
 * Dk and Dv are each 64, 128 or 256.  No workspace.  Returns GDN_OK or a
 * GDN_ERR_* code.
 */
GDN_API int gdn_decode_step(const void *q, const void *k, const void *v, const void *g,
                    const void *beta, const float *state_in, float *state_out,
                    void *y, int B, int Hk, int Hv, int Dk, int Dv, int dtype,
                    void *stream);

/* gdn_decode_step with input conventions `options` (GDN_OPT_* bits above). */
GDN_API int gdn_decode_step_ex(const void *q, const void *k, const void *v, const void *g,
                const void *beta, const float *state_in, float *state_out, void *y,
                int B, int Hk, int Hv, int Dk, int Dv, int dtype, void *stream,
                int options);

/*
 * Prefill for callers that cannot allocate device memory.  This entry point
 * has no counterpart in the source pages; it exists for the library's users.
 *
 * gdn_prefill needs a caller-allocated workspace.  Some callers cannot call
 * cudaMalloc: plug-ins that a host application hands raw device pointers but
 * no allocator of their own (and that must not take memory behind the host's
 * pool), and latency-critical paths that cannot afford cudaMalloc's implicit
 * device synchronisation.  They can call this instead.  It computes exactly
 * what gdn_prefill computes (same arguments and meaning, minus the workspace)
 * and allocates nothing: its scratch is a fixed array of
 * GDN_NOALLOC_SCRATCH_BYTES built into the library, one per CUDA context that
 * loads the library's kernels, held until that context is destroyed.
 *
 *   Limit: the problem's gdn_prefill_workspace_bytes(...) must not exceed
 *   GDN_NOALLOC_SCRATCH_BYTES; larger problems return GDN_ERR_NOALLOC_LIMIT
 *   with nothing enqueued.
 *   Set-up: the first call in each CUDA context (with that context current)
 *   looks up the array's device address once and remembers it for that
 *   context; make that first call before any stream capture.
 *   Sharing: every call in a context uses the same array, and the array
 *   keeps the previous call's contents (nothing in it needs to start at
 *   zero).  Two calls whose work overlaps on the GPU (different streams, no
 *   ordering between them) race on it and give undefined results; order them.
 * Returns GDN_OK or a GDN_ERR_* code, as gdn_prefill.
 */
#define GDN_NOALLOC_SCRATCH_BYTES (32u << 20)
GDN_API int gdn_prefill_noalloc(const void *q, const void *k, const void *v, const void *g,
                                const void *beta, const float *state_in, float *state_out,
                                void *y, int B, int T, int Hk, int Hv, int Dk, int Dv,
                                int chunk, int dtype, void *stream);

/*
 * Device-side health: every wait inside the tensor-core and TMA-fed kernels
 * (on an mbarrier fed by TMA or by the tensor core, or on a tile flag that
 * another CTA raises) is bounded; a wait that gives up
 * sets a device error word and the kernel returns early, leaving its outputs
 * unspecified.  This call synchronises the device, reads that word and
 * returns GDN_OK, GDN_ERR_DEVICE_TIMEOUT, or GDN_ERR_CUDA if it cannot be
 * read.  A non-zero `clear` resets the word.
 */
GDN_API int gdn_device_status(int clear);

/*
 * Failure-detection hook (for tests of gdn_device_status): enqueues on
 * `stream` one single-thread kernel that runs the library's two bounded waits
 * on things that never complete -- an mbarrier phase no thread arrives on,
 * then a device flag no code raises.  Each gives up after its limit (2 s), so
 * the kernel ends after about 4 s having set the device error word, and the
 * next gdn_device_status returns GDN_ERR_DEVICE_TIMEOUT.  It reads and writes
 * no caller memory and leaves the CUDA context usable.  Returns GDN_OK, or
 * GDN_ERR_CUDA if the launch failed.
 */
GDN_API int gdn_selftest_wait_timeout(void *stream);

/* A static, NUL-terminated description of a status code. */
GDN_API const char *gdn_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H_ */
