/*
 * qre.h -- C ABI of the quantized routed-expert MoE layer for GB300 (sm_103a).
 *
 * One routed mixture-of-experts layer: a sigmoid top-k router, a token->expert
 * dispatch through an expert slot (pointer) table, a fused dequant + SwiGLU
 * expert FFN over 4-bit group-quantized weights that live either in device
 * memory (HBM cache slots) or in pinned host memory read zero-copy, a shared
 * expert, and the routing-weighted combine.
 *
 * Sources.  The pages this library follows are serving recipes for
 * GLM-5.3-Flash with expert offload: "GLM-5.3-Flash EXL3 3.05bpw on 1x RTX PRO
 * 6000" (GPU expert cache, host-RAM streaming), "... on 1x RTX 3090" (RAM/NVMe
 * expert tiering), "... 2.05bpw on 2x RTX 5090" and the glm53-flash-offload
 * README.  They fix 288 routed experts, top-8 routing, a shared expert, expert
 * pointer tables rewritten in place, zero-copy reads of host-resident experts and
 * a ~1e-3 relative RMS error class per expert kernel.  They do not define the
 * router function, the weight codebook or any kernel; those are this library's.
 *
 * Conventions (all entry points)
 *   - Every pointer argument is a DEVICE pointer unless its comment says "host".
 *     Pinned host memory mapped into the device address space (cudaHostAlloc with
 *     cudaHostAllocMapped, or cudaHostRegister + device pointer) counts as a
 *     device pointer where a comment says "device or host-mapped".
 *   - The caller owns and allocates every buffer, including the workspace.  The
 *     library allocates no memory on any call and keeps no state apart from a
 *     per-device status word and a thread-local error message.
 *   - Calls are asynchronous on the given stream (NULL = the legacy default
 *     stream) and never synchronize with the host, except the two functions
 *     that read the device status word.  Dependent calls must share a stream.
 *   - Argument, shape and alignment errors are detected on the host before any
 *     launch and returned synchronously; nothing is launched then.  Launch
 *     failures return QRE_ERR_CUDA.  Conditions only visible on the device (a
 *     null slot pointer, a non-finite scale, a wait that ran out of time) are
 *     recorded in the device status word, and the kernel skips the affected
 *     work instead of faulting; read it with qre_read_device_status.
 *   - qre_last_error() returns the message of the last failing call made by
 *     the calling host thread.
 *   - Supported shapes: hidden and inter multiples of 128 and at most 4096;
 *     group in {32, 64, 128} dividing both; 1 <= n_experts <= 1024;
 *     1 <= top_k <= min(16, n_experts); 0 <= T <= 65536 / top_k.  T == 0 is a
 *     valid empty call that launches nothing.
 *   - Alignment: every array base must be 16-byte aligned.
 */
#ifndef QRE_H
#define QRE_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define QRE_API __attribute__((visibility("default")))
#else
#define QRE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream handle (cudaStream_t / CUstream). */
typedef struct CUstream_st* qre_stream_t;

typedef enum {
  QRE_OK = 0,
  QRE_ERR_INVALID_ARG = 1,   /* null pointer, negative size, k > E, ...            */
  QRE_ERR_UNSUPPORTED = 2,   /* shape outside the supported set                    */
  QRE_ERR_MISALIGNED = 3,    /* an array base is not 16-byte aligned               */
  QRE_ERR_WORKSPACE = 4,     /* workspace smaller than qre_workspace_size()        */
  QRE_ERR_CUDA = 5,          /* a CUDA runtime call or launch failed               */
  QRE_ERR_TIMEOUT = 6,       /* device status: a bounded wait ran out of time      */
  QRE_ERR_DEVICE_CHECK = 7   /* device status: a device-side check failed          */
} qre_status;

/* Device status word bits (qre_read_device_status). */
#define QRE_DEV_TIMEOUT       0x1   /* a pipeline wait gave up; results are invalid  */
#define QRE_DEV_NULL_SLOT     0x2   /* an active expert's slot has a null pointer    */
#define QRE_DEV_BAD_SCALE     0x4   /* quantize: a group scale was not finite        */
#define QRE_DEV_BAD_INDEX     0x8   /* an expert id outside [0, n_experts)           */
#define QRE_DEV_FP16_RANGE    0x10  /* prefill: an activation or h exceeded fp16     */

/* Layer shape.  H = hidden, I = expert intermediate, E = routed experts,
 * k = experts per token, G = quantization group along the reduction axis. */
typedef struct {
  int32_t hidden;
  int32_t inter;
  int32_t n_experts;
  int32_t top_k;
  int32_t group;
} qre_layer_shape;

/*
 * One expert slot: where an expert's packed weights are.  The slot table is a
 * DEVICE array of n_experts + 1 entries; entry n_experts is the shared expert.
 * It plays the role of the per-expert pointer tables that the RTX PRO 6000
 * recipe rewrites in place (config.expert_cache.mechanism): retargeting an
 * expert from a cache slot to host memory is a write of this struct.
 *
 * Weight format (packed 4-bit symmetric groups, fp16 scales), for a matrix
 * W [N, K] (N a multiple of 128, K of 64) with groups of G along K:
 *   s = fp16_RNE(max|w| / 7) (fp64 quotient), q = clamp(rint_half_even(w / s),
 *   -8, 7) (q = 0 when s == 0), nibble u = q + 8, even k in the low nibble of
 *   its byte; dequantized value (u - 8) * s.
 * Storage is tiled so that a warp reading 32 rows of one 32-column slice reads
 * 512 contiguous bytes:
 *   packed: 4096-byte chunks, chunk (n/128)*(K/64) + k/64; inside it byte
 *           2048*((k%64)/32) + 16*(n%128) + (k%32)/2
 *   scales: fp16 of (n, group g) at ((n/128)*(K/G) + g)*128 + n%128
 * The gate and up projections ([I, H] each) are stored as one [2I, H] matrix
 * whose rows alternate in blocks of 16 (16 gate rows, 16 up rows, ...).
 */
typedef struct {
  const uint8_t*  w_gate_up;  /* 2I x H packed (I*H bytes), device or host-mapped */
  const uint16_t* s_gate_up;  /* 2I x H/G fp16 scales, device or host-mapped      */
  const uint8_t*  w_down;     /* H x I packed (H*I/2 bytes), device or host-mapped */
  const uint16_t* s_down;     /* H x I/G fp16 scales, device or host-mapped       */
  uint32_t tier;              /* 0 = device memory (the decode kernels stage it
                                 through shared memory with cp.async), 1 =
                                 host-mapped (read with direct 16-byte loads over
                                 the host link); results are identical        */
  uint32_t reserved;          /* must be 0                                      */
} qre_slot;

/* Message of the last failing call on this host thread ("" if none). */
QRE_API const char* qre_last_error(void);

/* Short name of a status code. */
QRE_API const char* qre_status_string(qre_status status);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
QRE_API int32_t qre_version(void);

/*
 * Bytes of workspace that qre_route, qre_dispatch and qre_expert_ffn need for a
 * call with T tokens (the maximum over the three; one buffer serves all).
 * bytes: host pointer, written on success.  The workspace content need not be
 * initialised and is not preserved between calls.
 */
QRE_API qre_status qre_workspace_size(const qre_layer_shape* shape, int32_t T, size_t* bytes);

/*
 * Quantize an fp32 matrix into the packed format above (the same rule as the
 * slot table's comment).  This is the offline step that produces expert
 * weights; it is not part of the per-token path.
 *   w       [n_rows][k_dim] fp32, device
 *   packed  n_rows*k_dim/2 bytes, tiled as above, device (written)
 *   scales  n_rows*k_dim/group fp16 bits, tiled as above, device (written)
 * group in {32, 64, 128}; k_dim a positive multiple of group and of 64; n_rows
 * a multiple of 128 (0 is a no-op).
 * A non-finite scale sets QRE_DEV_BAD_SCALE in the device status word.
 */
QRE_API qre_status qre_quantize(int32_t n_rows, int32_t k_dim, int32_t group, const float* w,
                        uint8_t* packed, uint16_t* scales, qre_stream_t stream);

/*
 * Quantize one expert's gate and up projections (w_gate, w_up: [inter][hidden]
 * fp32, device) into the interleaved [2*inter][hidden] layout described at
 * qre_slot, tiled as described there: packed 2*inter*hidden/2 bytes and scales
 * 2*inter*hidden/group fp16 bits (device, written).  inter a positive multiple
 * of 64, hidden a positive multiple of group and of 64, group in {32, 64, 128}.
 * A non-finite scale sets QRE_DEV_BAD_SCALE.
 */
QRE_API qre_status qre_quantize_gate_up(int32_t inter, int32_t hidden, int32_t group, const float* w_gate,
                                        const float* w_up, uint8_t* packed, uint16_t* scales,
                                        qre_stream_t stream);

/*
 * Router: logits l = x W_r^T (fp32 accumulation: below 1024 tokens one fp32
 * FMA chain over ascending h per logit; from 1024 tokens on the tensor cores,
 * with W_r split into three bf16 parts whose sum is W_r exactly, so every
 * product is exact and only the accumulation order differs), scores s = sigmoid(l),
 * selection score s + bias (bias is selection-only; NULL = 0), the top_k experts
 * by selection score with ties to the lower id, written in ascending id order,
 * and weights w = s / sum(s over the selection).  Top-8 of 288: GLM-5.3-Flash
 * EXL3 3.05bpw on 1x RTX 3090 recipe, summary (each token takes 8 of the 288
 * experts of every layer);
 * the sigmoid/renormalise rule is this library's reading (the pages are silent).
 *   x_bf16    [T][H] bf16 bits, device
 *   w_router  [E][H] fp32, device
 *   bias      [E] fp32 or NULL, device
 *   topk_idx  [T][k] int32, device (written)
 *   topk_w    [T][k] fp32, device (written)
 *   workspace device, >= qre_workspace_size bytes
 */
QRE_API qre_status qre_route(const qre_layer_shape* shape, int32_t T, const uint16_t* x_bf16,
                     const float* w_router, const float* bias, int32_t* topk_idx,
                     float* topk_w, void* workspace, size_t workspace_bytes,
                     qre_stream_t stream);

/*
 * qre_route without a workspace: the same router as qre_route, with the same
 * bits below 1024 tokens (its logits always come from the fp32 FMA chains,
 * since the split weights of the tensor-core path need workspace), for callers
 * that cannot allocate device memory -- code that runs
 * inside a host framework which owns every device allocation, loops that must
 * not allocate once they run, or callers that only hold the input and output
 * buffers someone else gave them.  The pages have no counterpart; it is an
 * interface choice of this library.
 *   Scratch: a fixed array of 65,536 floats (256 KiB) inside the library, kept
 *   by every GPU that loads it until the process exits; T * n_experts must be at
 *   most 65,536 (QRE_ERR_UNSUPPORTED otherwise, nothing launched).
 *   The first call on each device looks up the array's device address with that
 *   device current; make that first call before any stream capture.  The
 *   address is kept for the life of the process: after cudaDeviceReset (or
 *   anything else that destroys the device's primary context) it no longer
 *   names the array, so do not call qre_route_noalloc on that device again in
 *   the same process.
 *   Every call shares the array: calls whose kernels may overlap on the GPU race
 *   and give wrong results; keep them on one stream or otherwise ordered.
 *   Nothing in the array has to start at zero.  No cudaMalloc, cudaFree or
 *   allocating library routine is called.
 * Arguments, layouts and errors are those of qre_route.
 */
QRE_API qre_status qre_route_noalloc(const qre_layer_shape* shape, int32_t T, const uint16_t* x_bf16,
                                     const float* w_router, const float* bias, int32_t* topk_idx,
                                     float* topk_w, qre_stream_t stream);

/*
 * Dispatch: deduplicate the picks into the expert union that all tokens share
 * (glm53-flash-offload README, "Elastic CLOCK expert cache": a one-block kernel
 * dedups the router picks; "Batched decode": streams share the per-layer expert
 * union).  For the T*k picks p = t*k + j:
 *   counts   [E] int32     picks per expert
 *   offsets  [E+1] int32   exclusive prefix sum of counts
 *   perm     [T*k] int32   pick ids sorted stably by (expert, p)
 *   inv_perm [T*k] int32   inv_perm[perm[q]] = q
 *   active   [E] int32     experts with counts > 0, ascending (first n_active valid)
 *   n_active [1] int32     number of active experts (stays on the device)
 * All outputs device, written.  topk_idx [T][k] int32 device: each row must hold
 * distinct ids in [0, E); an id outside that range sets QRE_DEV_BAD_INDEX and is
 * dropped.  Results are deterministic.
 */
QRE_API qre_status qre_dispatch(const qre_layer_shape* shape, int32_t T, const int32_t* topk_idx,
                        int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv_perm,
                        int32_t* active, int32_t* n_active, void* workspace,
                        size_t workspace_bytes, qre_stream_t stream);

/*
 * qre_route followed by qre_dispatch in one call, with the same outputs (bit
 * for bit) and arguments.  For one token the top-k selection and the dispatch
 * share one single-CTA kernel, one dependent launch less on the way to the
 * expert FFN; other T runs the two calls' kernels.  The workspace must hold
 * qre_workspace_size bytes.
 */
QRE_API qre_status qre_route_dispatch(const qre_layer_shape* shape, int32_t T, const uint16_t* x_bf16,
                                      const float* w_router, const float* bias, int32_t* topk_idx, float* topk_w,
                                      int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv_perm,
                                      int32_t* active, int32_t* n_active, void* workspace, size_t workspace_bytes,
                                      qre_stream_t stream);

/*
 * Expert FFN: for every active expert e and each of its picks, and for the
 * shared expert (slot n_experts) over all T tokens,
 *   o = W_down (silu(W_gate x) * (W_up x)),
 * with weights dequantized on the fly from the slot table (the fused MoE kernel
 * of the glm53-flash-offload README, "Quality" section: ~1e-3 relative RMS per
 * expert is the error class; host-resident experts are read zero-copy as in the
 * README's "Zero-copy home").
 *   x_bf16      [T][H] bf16 bits, device
 *   slots       [E+1] qre_slot, device
 *   offsets, perm, active, n_active: from qre_dispatch, device
 *   expert_out  [T*k + T][H] fp32, device (written): row q < T*k is the output
 *               of pick perm[q] (unweighted), row T*k + t the shared expert's
 *               output for token t.
 * T <= 8 runs the bandwidth-bound decode kernels: for group 128 the weights as
 * exact FP8 codes and the activations as sums of FP8 terms (x: two, exact for
 * bf16 unless an element is below 2^-13 of its 128-group's largest; h: four,
 * about 16 significant bits), exact products, fp32 accumulation; for groups 32
 * and 64 exact fp16 codes times x split into two fp16 parts.  Larger T runs
 * the grouped-GEMM path (fp16 operands, fp32 accumulation).
 */
QRE_API qre_status qre_expert_ffn(const qre_layer_shape* shape, int32_t T, const uint16_t* x_bf16,
                          const qre_slot* slots, const int32_t* offsets, const int32_t* perm,
                          const int32_t* active, const int32_t* n_active, float* expert_out,
                          void* workspace, size_t workspace_bytes, qre_stream_t stream);

/*
 * The expert FFN in two parts that may run concurrently on two streams: the
 * routed experts (qre_expert_ffn_routed, which needs the dispatch results) and
 * the shared expert (qre_expert_ffn_shared, which needs only x, so it can start
 * while the router and the dispatch run -- the glm53-flash-offload README's
 * "Decode kernels" bullet moves the shared expert to a side stream).  Together
 * they write exactly what one qre_expert_ffn call writes, with the same bits
 * (every expert row is computed by the same arithmetic whichever launch or CTA
 * computes it), so the combine order and the layer output do not change.
 *   qre_expert_ffn_routed: arguments as qre_expert_ffn; writes expert_out rows
 *     0 .. T*k-1; workspace >= qre_workspace_size bytes.
 *   qre_expert_ffn_shared: writes expert_out rows T*k .. T*k+T-1 (the shared
 *     expert's output per token) from x and slots[n_experts]; workspace: its own
 *     buffer of at least qre_shared_workspace_size bytes (not the one the router,
 *     the dispatch or the routed part use while it runs).
 */
QRE_API qre_status qre_expert_ffn_routed(const qre_layer_shape* shape, int32_t T, const uint16_t* x_bf16,
                                         const qre_slot* slots, const int32_t* offsets, const int32_t* perm,
                                         const int32_t* active, const int32_t* n_active, float* expert_out,
                                         void* workspace, size_t workspace_bytes, qre_stream_t stream);
QRE_API qre_status qre_expert_ffn_shared(const qre_layer_shape* shape, int32_t T, const uint16_t* x_bf16,
                                         const qre_slot* slots, float* expert_out, void* workspace,
                                         size_t workspace_bytes, qre_stream_t stream);
/* Bytes of workspace qre_expert_ffn_shared needs for T tokens (bytes: host). */
QRE_API qre_status qre_shared_workspace_size(const qre_layer_shape* shape, int32_t T, size_t* bytes);

/*
 * Combine: y[t] = sum_j topk_w[t][j] * expert_out[inv_perm[t*k + j]] +
 * expert_out[T*k + t], accumulated in fp32 in ascending j (ascending expert
 * id), the shared term last.  The fp32 partial sums are added after the
 * experts, as the glm53-flash-offload README's "CPU tier" bullet does.
 *   expert_out [T*k + T][H] fp32, topk_w [T][k] fp32, inv_perm [T*k] int32: device
 *   y_f32  [T][H] fp32, device (written)
 *   y_bf16 [T][H] bf16 bits or NULL, device (written): round-to-nearest-even
 *          of y_f32.
 */
QRE_API qre_status qre_combine(const qre_layer_shape* shape, int32_t T, const float* expert_out,
                       const float* topk_w, const int32_t* inv_perm, float* y_f32,
                       uint16_t* y_bf16, qre_stream_t stream);

/*
 * Expert cache, manager step (one CTA, stream-ordered, no host sync).  Per layer
 * and call, after qre_dispatch: the LFU scores decay, every miss takes the
 * lowest-scoring cache slot that this call does not use, and `table` (the slot
 * table qre_expert_ffn reads) is rewritten in place -- the RTX PRO 6000 recipe's
 * config.expert_cache.mechanism (decay 0.995 there).
 *   n_slots      number of cache slots S (1 <= S <= 1024)
 *   decay        score decay per call, e.g. 0.995
 *   active, n_active   this call's expert union, from qre_dispatch (device)
 *   scores       [E] fp32 (device, read-write); scores[e] = fp32(fp32(scores[e] *
 *                decay) + [e used by this call])
 *   expert_slot  [E] int32 (device, read-write): slot of e, -1 not cached, -2 static
 *   slot_expert  [S] int32 (device, read-write): expert in slot s, -1 empty
 *   home         [E+1] qre_slot (device): where each expert lives when it is not
 *                cached (pinned host memory, tier 1) -- never dereferenced here
 *   slot_mem     [S] qre_slot (device): the HBM addresses of the slots (tier 0)
 *   table        [E+1] qre_slot (device, rewritten): admitted experts -> their
 *                slot, evicted experts -> home
 *   copy_list    [2 * max_copies] int32 (device, written): (expert, slot) pairs
 *   n_copies     [1] int32 (device, written): admissions of this call
 * Misses are handled in ascending expert id; the victim is the candidate slot
 * with the lowest score of its current expert (empty slots first), ties to the
 * lowest slot index; a miss with no candidate stays host-resident this call.
 * A call admits at most max_copies experts: once the copy list is full, the
 * remaining misses of the call also stay host-resident (their table entries
 * unchanged), so every slot the table points at holds its expert's weights
 * after qre_cache_copy.
 */
QRE_API qre_status qre_cache_update(const qre_layer_shape* shape, int32_t n_slots, float decay,
                                    const int32_t* active, const int32_t* n_active, float* scores,
                                    int32_t* expert_slot, int32_t* slot_expert, const qre_slot* home,
                                    const qre_slot* slot_mem, qre_slot* table, int32_t* copy_list,
                                    int32_t* n_copies, int32_t max_copies, qre_stream_t stream);

/*
 * Expert cache, miss copy: copies each admitted expert's four arrays from
 * home[e] (pinned host memory, read over the host link) to slot_mem[s] (HBM),
 * reading the number of copies on the device (no host sync).  Arguments as in
 * qre_cache_update; all device.
 */
QRE_API qre_status qre_cache_copy(const qre_layer_shape* shape, const qre_slot* home, const qre_slot* slot_mem,
                                  const int32_t* copy_list, const int32_t* n_copies, int32_t max_copies,
                                  qre_stream_t stream);

/*
 * Prefill staging: a prefill chunk touches nearly every expert of a layer, so
 * the experts that live in host memory are copied into HBM one layer ahead on
 * a copy stream, and the FFN reads the staged copies (the RTX PRO 6000
 * recipe's config.expert_cache.mechanism, prefill staging; the
 * glm53-flash-offload README, "Prefill staging").  For each entry e of the
 * layer's slot table with tier 1, in ascending e while staging slots remain,
 * the expert's four arrays are copied with cudaMemcpyAsync (the copy engines,
 * leaving the SMs to the computation) into the next staging slot, and the staged
 * table's entry e points there (tier 0); every other entry is copied as it is.
 *   host_table    [E+1] qre_slot, HOST: the layer's table
 *   host_staging  [n_staging] qre_slot, HOST: the staging slots (device memory, tier 0)
 *   host_out      [E+1] qre_slot, HOST, written by this call and uploaded on the
 *                 stream: keep it unchanged until the stream has passed the call
 *                 (pinned memory keeps the upload asynchronous)
 *   table_out     [E+1] qre_slot, DEVICE: the staged table (written on the stream)
 *   n_staged      host int32: experts staged (the rest of tier 1 stays host-mapped)
 * The staging slots must not be in use by a kernel that runs concurrently (use
 * two staging areas to stage layer l+1 while layer l computes).  Works inside
 * CUDA graph capture (the copies and the upload become graph nodes).
 */
QRE_API qre_status qre_stage_experts(const qre_layer_shape* shape, const qre_slot* host_table,
                                     const qre_slot* host_staging, int32_t n_staging, qre_slot* host_out,
                                     qre_slot* table_out, int32_t* n_staged, qre_stream_t stream);

/*
 * Bandwidth probe: one streaming read of `bytes` bytes at src (device memory,
 * or pinned host memory mapped into the device address space, read zero-copy
 * the way host-resident experts are read), 16-byte loads with several in flight
 * per thread over 4 CTAs per SM.  Time it with events on `stream` to get the
 * copy-free read rate of device memory or of the host link.  src 16-byte
 * aligned, bytes a positive multiple of 16; sink: one device uint32 the kernel
 * may write (it keeps the loads from being removed).
 */
QRE_API qre_status qre_read_probe(const void* src, size_t bytes, uint32_t* sink, qre_stream_t stream);

/*
 * Checks a HOST copy of a slot table before it is uploaded: every pointer
 * non-null and 16-byte aligned, reserved == 0, tier in {0, 1}, tier-0
 * pointers in device memory and tier-1 pointers in host memory that the
 * device can read.  host_slots: host array of n_experts + 1 entries.
 */
QRE_API qre_status qre_validate_slots(const qre_layer_shape* shape, const qre_slot* host_slots);

/*
 * Decode expert FFN with host-mapped experts in the slot table (the
 * expert-cache layout): every call after this one, process-wide, cuts the
 * decode kernels' work ranges at equal cost with a 128-row unit of a
 * host-mapped expert counted as `cost` units of device memory (it streams over
 * the host link at a fraction of the rate), so host-resident experts spread
 * over more SMs.  0 or 1 (the default) cuts at equal unit counts, the right
 * choice when every expert is in device memory.  cost in [0, 64].  Results are
 * the same bits either way.  A CUDA graph keeps the value in force when it was
 * captured.  On a GB300 with 100 of 288 experts in pinned host memory read over
 * a ~211 GB/s link, 3 gave the shortest decode FFN of the values 2 to 6.
 */
QRE_API qre_status qre_set_host_unit_cost(int32_t cost);

/*
 * Test hook for the bounded waits' give-up path (failure handling without a
 * GPU fault).  Every kernel of this library bounds its pipeline waits; one that
 * runs out of time sets QRE_DEV_TIMEOUT, makes the CTA's other waits give up,
 * lets the tensor core finish what was issued, frees its tensor memory and
 * returns, so the context stays usable and the next call is unaffected.
 *   wait_limit_ns  limit of the pipeline waits of later launches (process-wide),
 *                  0 restores the default of one second; at most one second.
 *   stall_ns       when non-zero, later expert-FFN launches delay one warp of
 *                  one CTA (the decode kernels: the CTA that owns the first
 *                  unit of work; the grouped GEMM: CTA 0's token loads) by this
 *                  long before it signals its first pipeline stage (at most
 *                  100 ms), so that a wait with a shorter limit runs out; 0
 *                  turns it off.
 * Results of calls made while a wait runs out are invalid.  Not for production
 * use; a CUDA graph keeps the values in force when it was captured.
 */
QRE_API qre_status qre_debug_wait_test(uint64_t wait_limit_ns, uint64_t stall_ns);

/*
 * Synchronizes the stream, then writes the current device's status word
 * (QRE_DEV_* bits, 0 = clean) to *status (host).  qre_clear_device_status
 * resets it to 0 (also synchronizing the stream).
 */
QRE_API qre_status qre_read_device_status(qre_stream_t stream, int32_t* status);
QRE_API qre_status qre_clear_device_status(qre_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* QRE_H */
