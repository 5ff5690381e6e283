/*
 * psf.h -- C ABI of the packed-sequence flash-attention library (libpsf.so).
 *
 * Exact softmax attention over packed variable-length sequences on one GB300
 * (sm_103a): forward returning out and an fp32 log-sum-exp, backward from
 * caller-supplied out/lse returning dQ and dK/dV reduced to the KV heads, and
 * the doc-ids -> varlen-segment builder that feeds them.
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Pointers are DEVICE pointers owned by the caller; the library allocates
 *    nothing. Outputs and workspaces are caller-allocated. Tensor base pointers
 *    must be 16-byte aligned (a TMA requirement).
 *  - Strides: the attention calls take `strides`, NULL for the layout's
 *    contiguous strides, else an int64 array of element strides, three per
 *    tensor in the order (batch, head, row), tensors in the order each call
 *    lists. The head dim is always contiguous. A stride of a dimension of
 *    extent 1 (the batch of a packed THD tensor, a single head or row) is
 *    ignored; every other one must be a positive multiple of 8 elements
 *    (16 bytes) below 2^38, and an output's strides must not make it overlap
 *    itself (PSF_EINVAL otherwise). lse stays contiguous.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *    Every call is asynchronous on that stream.
 *  - Return value: PSF_OK (0) after a successful launch, or a negative code.
 *    No exception crosses the ABI. psf_last_error() gives a message for the
 *    last failing call on the calling thread.
 *  - Kernel-side faults in the caller's data (bad segment arrays) and pipeline
 *    waits that ran out are recorded in a per-device status word that
 *    psf_device_status() returns after synchronising the device.
 *  - dtype: bf16 or fp16 inputs and outputs (`out`, `dq`, `dk`, `dv`), chosen
 *    per call by a PSF_DTYPE_* argument; lse and the row-dot Delta are fp32.
 *  - Head dims (Dqk, Dv) supported: (64,64), (128,128), (192,128), (512,512).
 *    The (512,512) backward launches four-CTA thread-block clusters, as many
 *    as the device holds at once; where it holds none (PSF_ECUDA).
 *  - GQA: Hq % Hkv == 0; query head h uses KV head h / (Hq / Hkv).
 *  - Causal masks are aligned to the bottom-right corner of each segment
 *    (dense: of the Nq x Nk matrix): local query i of a segment with m queries
 *    and n keys sees local key j iff j <= i + (n - m).
 *  - window_left > 0 is a left window that counts the current token: key j is
 *    visible only if j >= i + (n - m) - window_left + 1. window_left < 0 (for
 *    example INT32_MIN, the pages' "no window" sentinel) means unbounded;
 *    window_left == 0 is rejected with PSF_EINVAL.
 *  - Query rows covered by no segment, and rows that see no key, get out = 0
 *    and lse = -inf; the backward treats lse = -inf as zero probability.
 *  - scale must be finite and > 0.
 */
#ifndef PSF_H_
#define PSF_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PSF_OK 0
#define PSF_EINVAL (-1)        /* bad argument: shape, null pointer, alignment, window == 0, scale */
#define PSF_EUNSUPPORTED (-2)  /* no kernel for this head-dim pair, or the device is not sm_103 */
#define PSF_ECUDA (-3)         /* a CUDA runtime call (launch, tensor-map encode) failed */
#define PSF_EDEVICE_ARGS (-4)  /* kernel-side validation rejected the segment arrays */
#define PSF_ETIMEOUT (-5)      /* a pipeline wait inside a kernel exceeded its limit */
#define PSF_EWORKSPACE (-6)    /* workspace pointer null or smaller than the size query */

/* Tensor layouts accepted by the varlen calls. */
#define PSF_LAYOUT_THD 0  /* packed [T, H, D]; lse [H, T]                                */
#define PSF_LAYOUT_BHSD 1 /* batched [B, H, S, D]; lse [B, H, S]; rows are b * S + s     */

/*
 * Element type of the 16-bit tensors of a call (q, k, v, out, dout, dq, dk, dv,
 * merge operands); one type per call. lse, Delta and every accumulator stay
 * fp32.                     [ffpa_attention page, module docstring: the op
 *                            takes bf16 and fp16 inputs]
 */
#define PSF_DTYPE_BF16 0
#define PSF_DTYPE_F16 1

/* Message for the last failing call on this thread (never NULL). */
const char* psf_last_error(void);

/* 1 if the current device is an sm_103 GPU this library was built for, else 0. */
int psf_device_supported(void);

/*
 * Synchronise the current device and return the first kernel-side status
 * recorded since the last clear: PSF_OK, PSF_EDEVICE_ARGS or PSF_ETIMEOUT.
 * clear != 0 resets it to PSF_OK.
 */
int psf_device_status(int clear);

/* Upper bound, in nanoseconds, of every pipeline wait inside the kernels
 * (default 2e9, or $PSF_WAIT_LIMIT_NS when set at load time). */
void psf_set_wait_limit_ns(uint64_t ns);

/*
 * Check of the failure path every pipeline wait takes, without a fault: one
 * CTA of 64 threads on `stream` whose warp 0 waits on an mbarrier that expects
 * one arrival. With arrive != 0 warp 1 arrives and the kernel ends at once;
 * with arrive == 0 nothing arrives, the wait gives up after the current wait
 * limit (psf_set_wait_limit_ns), records PSF_ETIMEOUT in the status word that
 * psf_device_status() reads, and the kernel returns normally, leaving the
 * context usable. Returns PSF_OK once launched (PSF_EUNSUPPORTED on another
 * device, PSF_ECUDA if the launch fails).
 */
int psf_check_pipeline_wait(int arrive, void* stream);

/*
 * Kernel timing for profiling. psf_kernel_timing(1) clears the record and
 * starts it: from then on every attention call records two CUDA events on its
 * stream, immediately before and after its main kernel (kind 0: forward main
 * kernel, kind 1: backward main kernel). psf_kernel_timing(0) stops recording.
 * psf_kernel_times_ms() waits for the recorded events of `kind` and returns
 * their summed device time in *total_ms and their number in *launches.
 * Calls made while a stream capture is active record the pair as event-record
 * nodes of the captured graph: each replay of the graph re-records them, and
 * psf_kernel_times_ms() after a replay returns that replay's kernel times.
 */
int psf_kernel_timing(int enable);
int psf_kernel_times_ms(int kind, double* total_ms, int* launches);

/*
 * Workspace sizes in bytes. total_q_rows / total_k_rows count the flattened
 * query / key rows (T for THD, B * S for BHSD); nseg is the number of segments
 * (or the capacity passed to the builder).
 */
size_t psf_attn_fwd_workspace_size(int64_t total_q_rows, int nseg);
size_t psf_attn_bwd_workspace_size(int64_t total_q_rows, int64_t total_k_rows, int nseg, int Hq, int Hkv, int Dqk,
                                   int Dv);

/*
 * Varlen forward.           [ffpa_attention page, `_ffpa_varlen_fwd`: packed THD
 *                            inputs, cu_q/cu_k/max_q/max_k/scale/causal, returns
 *                            (out[T,Hq,D], lse[Hq,T]); left window per the
 *                            attention utils page, `window_size`]
 *  q [Tq,Hq,Dqk], k [Tk,Hkv,Dqk], v [Tk,Hkv,Dv] -> out [Tq,Hq,Dv], lse [Hq,Tq]
 *  (layout PSF_LAYOUT_THD), or the BHSD forms with Tq = B*Sq, Tk = B*Sk and
 *  lse [B,Hq,Sq] (layout PSF_LAYOUT_BHSD; a segment must not cross a batch row).
 *  cu_q / cu_k: int32 [nseg+1] device arrays of exclusive prefix sums over the
 *  flattened rows; segment s pairs queries [cu_q[s], cu_q[s+1]) with keys
 *  [cu_k[s], cu_k[s+1]); zero-length segments are allowed.
 *  dev_meta: nullable int32[3] device array {nseg, max_q, max_k} written by
 *  psf_build_doc_segments; when given, the segment count and maxima are read
 *  from it on the device and `nseg` is only the capacity of cu_q/cu_k.
 *  max_q / max_k: the longest segment lengths (ignored when dev_meta is given);
 *  a longer segment is a PSF_EDEVICE_ARGS device status.
 *  softcap: 0 (off), or c > 0: every logit z = scale * q . k becomes
 *  c * tanh(z / c) before the mask and the softmax (lse is over the capped
 *  logits). Negative or non-finite values are PSF_EINVAL.
 *                           [ffpa_attention page, `ffpa_attention_forward`
 *                            softcap argument; the eager attention the page
 *                            falls back to for it caps the scaled scores so]
 *  flags: 0, or PSF_FWD_PACK_GQA: the G = Hq / Hkv query heads of a KV head
 *  share one 128-row tile (128 / G rows of each), so short segments fill the
 *  tile and K/V are loaded once for all G heads. Same results; it applies to
 *  head dims (64, 64) and (128, 128) with G in 2..16 dividing 128, and other
 *  shapes run one head per tile.
 *                           [ffpa_attention page, `_ffpa_varlen_fwd`: the
 *                            pack-GQA sentinel the pages fix off]
 *  Any other bit is PSF_EINVAL.
 *  strides: NULL, or 12 element strides (batch, head, row) of q, k, v, out;
 *  for THD the row stride steps tokens and the batch stride is ignored.
 *  workspace: psf_attn_fwd_workspace_size(Tq, nseg) bytes (enough for either flag).
 */
#define PSF_FWD_PACK_GQA 1
int psf_attn_varlen_fwd(const void* q, const void* k, const void* v, void* out, float* lse, const int32_t* cu_q,
                        const int32_t* cu_k, const int32_t* dev_meta, int nseg, int max_q, int max_k, int layout,
                        int dtype, int B, int Sq, int Sk, int Hq, int Hkv, int Dqk, int Dv, const int64_t* strides,
                        float scale, int causal, int32_t window_left, float softcap, int flags, void* workspace,
                        size_t ws_bytes, void* stream);

/*
 * Varlen forward that allocates nothing and takes no workspace.
 *                           [no counterpart on the pages: an addition of this
 *                            library for callers that cannot allocate]
 *  Some callers cannot call cudaMalloc on this path: runtimes that reserve all
 *  device memory up front and hand out nothing afterwards, plugin hosts that
 *  own every allocation, or code that must not touch the allocator while a
 *  step runs. This entry point behaves like psf_attn_varlen_fwd (same
 *  arguments minus strides, softcap, flags, workspace and ws_bytes: contiguous
 *  tensors, no softcap, one query head per tile, same results) but keeps its tile
 *  schedule in a fixed array in the library's device memory (852,736 bytes,
 *  held on every GPU that loads the library until the process exits).
 *  Limits: B * Sq <= PSF_NOALLOC_MAX_Q_ROWS and nseg <= PSF_NOALLOC_MAX_SEGMENTS;
 *  larger calls return PSF_EINVAL without launching anything.
 *  The first call on a device looks up that array's device address (with the
 *  device current); make that first call before any stream capture.
 *  Every call shares the one array and leaves its contents behind; the
 *  schedule kernel rewrites all of it that a call reads, so nothing needs
 *  clearing between calls. Calls whose kernels overlap on the GPU (different
 *  streams, or different host threads, without ordering between them) race on
 *  the array and must not be issued.
 */
#define PSF_NOALLOC_MAX_Q_ROWS (1 << 20)
#define PSF_NOALLOC_MAX_SEGMENTS 65536
int psf_attn_varlen_fwd_noalloc(const void* q, const void* k, const void* v, void* out, float* lse,
                                const int32_t* cu_q, const int32_t* cu_k, const int32_t* dev_meta, int nseg,
                                int max_q, int max_k, int layout, int dtype, int B, int Sq, int Sk, int Hq, int Hkv,
                                int Dqk, int Dv, float scale, int causal, int32_t window_left, void* stream);

/*
 * Varlen backward from caller-supplied out / lse.
 *                           [ffpa_attention page, `_ffpa_varlen_bwd`: "using the
 *                            caller-supplied out/lse. Returns (dq, dk, dv)"]
 *  Same layouts and segment rules as the forward. dout has the layout of out.
 *  dq has q's layout; dk / dv have k's / v's layout (Hkv heads: the gradients of
 *  the Hq / Hkv query heads sharing a KV head are summed on chip).
 *  Keys that no query sees get dk = dv = 0; query rows outside every segment
 *  get dq = 0.
 *  softcap: the forward's (0 = off); with c > 0, dS carries 1 - tanh^2(z / c).
 *  flags: 0, or PSF_BWD_PACK_GQA: each step takes the G = Hq / Hkv query heads
 *  of its KV head, 128 / G rows each (head dims up to 128 with G = 2 or 4 and
 *  no softcap; other calls take one head per step). Same results; for short segments,
 *  where one head's rows fill little of a 128-row step. Other bits: PSF_EINVAL.
 *  strides: NULL, or 24 element strides (batch, head, row) of q, k, v, out,
 *  dout, dq, dk, dv.
 *  workspace: psf_attn_bwd_workspace_size(Tq, Tk, nseg, Hq, Hkv, Dqk, Dv) bytes
 *  (holds the fp32 dQ accumulator, Delta = rowsum(dO * out), the tile schedule
 *  and, for head dims up to 128, the fp32 dK/dV partial sums of key tiles cut
 *  across SMs; its size grows with Tq, not with Tk beyond the schedule).
 */
int psf_attn_varlen_bwd(const void* dout, const void* q, const void* k, const void* v, const void* out,
                        const float* lse, void* dq, void* dk, void* dv, const int32_t* cu_q, const int32_t* cu_k,
                        const int32_t* dev_meta, int nseg, int max_q, int max_k, int layout, int dtype, int B, int Sq,
                        int Sk, int Hq, int Hkv, int Dqk, int Dv, const int64_t* strides, float scale, int causal,
                        int32_t window_left, float softcap, int flags, void* workspace, size_t ws_bytes,
                        void* stream);
#define PSF_BWD_PACK_GQA 1

/*
 * Dense forward on SDPA-layout tensors.
 *                           [ffpa_attention page, `_ffpa_dense_fwd`: [B,H,N,D]
 *                            inputs, returns (out[B,Hq,Nq,D], lse[B,Hq,Nq] fp32),
 *                            GQA and causal/non-causal handled internally;
 *                            fa4 page, `causal_fa4_attention`]
 *  q [B,Hq,Nq,Dqk], k [B,Hkv,Nk,Dqk], v [B,Hkv,Nk,Dv], out [B,Hq,Nq,Dv],
 *  lse [B,Hq,Nq]. Causal is bottom-right aligned when Nq != Nk.
 *  strides: NULL (contiguous [B,H,N,D]) or 12 element strides (batch, head,
 *  row) of q, k, v, out: for example a [B,N,H,D] tensor seen as [B,H,N,D]
 *  (strides N*H*D, D, H*D) is read in place.
 *  softcap, flags: as for psf_attn_varlen_fwd.
 *  workspace: psf_attn_fwd_workspace_size(B * Nq, B) bytes.
 */
int psf_attn_dense_fwd(const void* q, const void* k, const void* v, void* out, float* lse, int B, int Hq, int Hkv,
                       int Nq, int Nk, int Dqk, int Dv, const int64_t* strides, int dtype, float scale, int causal,
                       int32_t window_left, float softcap, int flags, void* workspace, size_t ws_bytes,
                       void* stream);

/*
 * Dense backward.           [ffpa_attention page, `_ffpa_dense_bwd`: returns
 *                            (dq, dk, dv) in [B,H,N,D], dK/dV reduced to Hkv]
 *  strides: NULL or 24 element strides (batch, head, row) of q, k, v, out,
 *  dout, dq, dk, dv.
 *  softcap, flags: as for psf_attn_varlen_bwd.
 *  workspace: psf_attn_bwd_workspace_size(B * Nq, B * Nk, B, Hq, Hkv, Dqk, Dv) bytes.
 */
int psf_attn_dense_bwd(const void* dout, const void* q, const void* k, const void* v, const void* out,
                       const float* lse, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int Nq, int Nk,
                       int Dqk, int Dv, const int64_t* strides, int dtype, float scale, int causal,
                       int32_t window_left, float softcap, int flags, void* workspace, size_t ws_bytes,
                       void* stream);

/*
 * Doc ids -> varlen segments, on the GPU.
 *                           [fa4 page, module docstring bullets 1-3,
 *                            `_varlen_segments`, `_varlen_layout`]
 *  kv_doc_ids: int32 [B, Sk] document ids (1-based, 0 = padding) of all keys.
 *  The local query shard is [q_global_start, q_global_start + q_length) of
 *  every row. Every maximal run of equal id (padding runs included) is split at
 *  the end of the shard; each piece contributes its overlap with the shard as
 *  queries and all of its tokens as keys; pieces without queries become
 *  zero-query segments, so the key segments tile the flattened [B * Sk] rows
 *  and the query segments tile [B * q_length]. Segments are listed row-major.
 *  Outputs: cu_q, cu_k (int32, capacity + 1 entries each, prefix sums),
 *  dev_meta int32[3] = {nseg, max_q, max_k}, and seg_is_pad (nullable, uint8
 *  [capacity]: 1 for a segment cut from a padding run).
 *  flags: 0, or PSF_SEGMENTS_SKIP_PAD: every piece cut from a padding run is
 *  written as two segments, its queries with no keys, then its keys with no
 *  queries. The attention then gives padding queries out = 0 and lse = -inf by
 *  itself (no psf_pad_fixup needed) and computes no padding-vs-padding pairs;
 *  dK/dV of padding keys come out 0. Any other bit is PSF_EINVAL.
 *                           [fa4 page, `document_causal_fa4_attention`: padding
 *                            queries are zero; cp_attention page,
 *                            `_build_packed_ring_segments`: pad query rows zeroed]
 *  capacity: room in cu_q / cu_k; B * Sk + B always suffices without flags,
 *  2 * (B * Sk + B) with PSF_SEGMENTS_SKIP_PAD. Too small a capacity is a
 *  PSF_EDEVICE_ARGS device status (dev_meta[0] is then 0).
 *  Requires 0 <= q_global_start, q_global_start + q_length <= Sk.
 */
#define PSF_SEGMENTS_SKIP_PAD 1
int psf_build_doc_segments(const int32_t* kv_doc_ids, int B, int Sk, int q_length, int q_global_start,
                           int32_t* cu_q, int32_t* cu_k, int capacity, int32_t* dev_meta, uint8_t* seg_is_pad,
                           int flags, void* stream);

/*
 * Dense-kernel eligibility of one ring chunk, on the GPU.
 *                           [cp_attention page, `_build_packed_ring_segments`
 *                            (the dense_local / dense_cross flags and pad_rows)
 *                            and `_chunk_dense_eligible`; the row predicates:
 *                            one document and no padding, or the real tokens
 *                            one document that forms a contiguous prefix with
 *                            padding only as a trailing suffix]
 *  kv_doc_ids: int32 [B, S] (1-based ids, 0 = padding); the query shard is
 *  [q_start, q_start + q_length) and the key chunk [k_start, k_start + k_length)
 *  of every row. Writes flags, a device int32[2], 1 = eligible:
 *   flags[0] (local role, causal): the chunk ends where the shard ends and
 *     contains it, and in every row the chunk's real tokens are one document
 *     forming a prefix (padding only as a suffix; an all-padding row counts).
 *     psf_attn_dense_fwd/bwd (causal) on the raw [B, H, N, D] shard and chunk,
 *     then psf_pad_fixup on the shard's ids, give the document-causal result.
 *   flags[1] (cross role, non-causal): the chunk lies before the shard, in
 *     every row [k_start, q_start) is one document d > 0 without padding, and
 *     the shard starts with d and holds no other document (padding only as a
 *     suffix). The non-causal dense kernels, then psf_pad_fixup, give the
 *     result of the psf_build_cross_segments segments.
 *  Errors: PSF_EINVAL when the shard or the chunk leaves the row.
 */
int psf_chunk_dense_flags(const int32_t* kv_doc_ids, int B, int S, int q_start, int q_length, int k_start,
                          int k_length, int32_t* flags, void* stream);

/*
 * Zero the padding queries of a document-causal result: rows whose query
 * document id is 0 get out = 0 and lse = -inf.
 *                           [fa4 page, `document_causal_fa4_attention`:
 *                            padding queries give zero output; cp_attention
 *                            page: rows that take no part get lse = -inf]
 *  q_doc_ids: int32 [B, Lq]; out / lse in `layout` with S = Lq.
 */
int psf_pad_fixup(void* out, float* lse, const int32_t* q_doc_ids, int layout, int B, int Lq, int Hq, int Dv,
                  void* stream);

/*
 * Merge two partial attention results computed over disjoint key sets.
 *                           [cp_attention page, "-inf-safe online-softmax merge"]
 *  l = logaddexp(l1, l2); o = o1 * exp(l1 - l) + o2 * exp(l2 - l), in fp32. A
 *  row with both inputs -inf gives o = 0, l = -inf (never NaN).
 *  o1, o2: dtype [T, H, D]; l1, l2: fp32 [H, T] (PSF_LAYOUT_THD only).
 *  Outputs: o_f32 (nullable) fp32 [T,H,D], o_bf16 (nullable) dtype [T,H,D],
 *  l fp32 [H,T]. Outputs may alias neither input.
 */
int psf_lse_merge(const void* o1, const float* l1, const void* o2, const float* l2, float* o_f32, void* o_bf16,
                  float* l, int T, int H, int D, int dtype, void* stream);

/*
 * Cross-chunk segments of a query shard against an earlier key chunk, on the
 * GPU (the one-device core of the ring decomposition).
 *                           [cp_attention page, `_build_packed_ring_segments`:
 *                            for each document present in both the query shard
 *                            and the KV chunk, its query tokens are paired with
 *                            its key tokens as one segment, cu_q[i] pairing
 *                            cu_k[i]; the chunk before the shard runs without a
 *                            causal mask]
 *  kv_doc_ids: int32 [B, S] document ids (1-based, 0 = padding, no document).
 *  The shard is [q_start, q_start + q_length) and the chunk
 *  [k_start, k_start + k_length) of every row, with the chunk before the shard
 *  (k_start + k_length <= q_start); the shard's queries and the chunk's keys are
 *  packed row-major as B * q_length and B * k_length rows. Since documents are
 *  contiguous runs, only the run holding position q_start can be shared. Each
 *  row gives three segments: (no queries x the chunk keys before the shared
 *  run), (the run's shard queries x its chunk keys), (the remaining shard
 *  queries x no keys); with nothing shared the middle one is empty.
 *  Outputs: cu_q, cu_k int32 [3 B + 1]; dev_meta int32[3] = {3 B, max_q, max_k}.
 *  Run the chunk with psf_attn_varlen_fwd/bwd, causal = 0: shard queries outside
 *  the shared run get out = 0, lse = -inf, dq = 0.
 *  Errors: PSF_EINVAL when the chunk does not lie before the shard.
 */
int psf_build_cross_segments(const int32_t* kv_doc_ids, int B, int S, int q_start, int q_length, int k_start,
                             int k_length, int32_t* cu_q, int32_t* cu_k, int32_t* dev_meta, void* stream);

/*
 * Merge one key chunk's result into a running result, in place, on the query
 * rows that took part in the chunk.
 *                           [cp_attention page, the in-place live-row merge of
 *                            a varlen chunk into the running accumulators at its
 *                            rows only, with the online-softmax merge]
 *  Live rows: the query rows of segments (cu_q, cu_k) that have at least one
 *  key. On those rows l = logaddexp(l_acc, l_new) and o = o_run exp(l_acc - l)
 *  + o_new exp(l_new - l) (both -inf gives o = 0, l = -inf); other rows are not
 *  touched. Running output: o_acc fp32 [T, H, D] (nullable) and/or o_run dtype
 *  [T, H, D] (nullable), read from o_acc when given, written to both; l_acc fp32
 *  [H, T] in place. o_new dtype [T, H, D], l_new fp32 [H, T]. No two of o_acc,
 *  o_run, o_new alias one another, nor l_acc and l_new.
 *  Segments: nseg (or dev_meta[0], capped at nseg, when dev_meta is given).
 */
int psf_lse_merge_live_rows(float* o_acc, void* o_run, float* l_acc, const void* o_new, const float* l_new,
                            const int32_t* cu_q, const int32_t* cu_k, const int32_t* dev_meta, int nseg, int T, int H,
                            int D, int dtype, void* stream);

/*
 * Add one key chunk's query gradient into the running one on the query rows
 * that took part in the chunk.
 *                           [cp_attention page, the in-place grad scatter-add
 *                            of a chunk's packed gradient into the full one]
 *  dst += src on the live rows of (cu_q, cu_k) (as in psf_lse_merge_live_rows),
 *  dtype [T, H, D] both, added in fp32 and rounded once; other rows untouched.
 *  dst and src do not alias.
 */
int psf_grad_add_live_rows(void* dst, const void* src, const int32_t* cu_q, const int32_t* cu_k,
                           const int32_t* dev_meta, int nseg, int T, int H, int D, int dtype, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PSF_H_ */
