/*
 * kvq.h -- decode-time attention over a compressed (mixed-precision) VLM KV
 * cache, for one NVIDIA GB300 (sm_103a).  C ABI; no CUDA or torch types.
 *
 * What the library computes (sources, by page and section):
 *   - "VLM_KV_Quantization" (nuiw.github.io), section 2: each layer stores a
 *     K/V cache of shape [B, H_kv, T, D] (e.g. [1, 4, T, 128] for
 *     LLaVA-OneVision-7B, GQA with 28 query heads over 4 KV heads); K is
 *     stored after RoPE.  Intro checklist and section 1: only the historical
 *     cache is compressed, the current/question tokens never are, INT8/INT4/
 *     INT2 must really cost that many bits per value.  Section 4: K and V get
 *     their own bit-widths at the same tokens and group size.
 *   - HeadGuard news brief (jiinsi.com), key ideas: about 1/8 of the physical
 *     KV heads keep their image K (and V) in bf16; composable with any
 *     low-bit quantiser.
 *   - WSVD summary (gist.science 2604.02570), section 2.라: reconstruct K/V on
 *     chip inside a flash-decoding pipeline (QK, softmax, PV fused) and never
 *     write the reconstructed tensors back to device memory.
 *
 * Readings where the pages are silent:
 *   quantiser = group-wise asymmetric min-max along D, groups of G consecutive
 *   elements, scale s = fp16((max - min) / (2^b - 1)), zero z = fp16(min + 0),
 *   code = clamp(rint_half_even((x - z) / s), 0, 2^b - 1) in fp32 with the
 *   stored fp16 s and z (code 0 if s == 0); dequantised value = code * s + z.
 *   bits == 16 keeps bf16.  Query head hq reads KV head hq / (H_q / H_kv).
 *
 * Storage order of a packed row (this library's own layout; the pages only
 * ask that a b-bit code really take b bits).  The D = 128 codes of one
 * position of one head fill 128 slots, slot j at bit b * (j mod (32/b)) of
 * uint32 word j / (32/b) (little-endian).  Element d sits in slot
 *   K rows, d = 32P + 8t + 4e + i (P, t, i in [0,4), e in {0,1}):
 *     b = 2:  32t + 16*floor(i/2) + 8e + c,  c = {{4,7},{3,6},{2,5},{0,1}}[P][i mod 2]
 *     b = 4:  32t + 8i + 4e + P
 *     b = 8:  32t + 4*(2P + floor(i/2)) + 2e + (i mod 2)
 *   V rows, d = 16m + 8r + n (m, n in [0,8), r in {0,1}), every b:
 *     16n + 2m + r
 * so that each tensor-core operand register of the decode kernel comes out
 * of one masked word.  The scale/zero row of a packed row
 * holds fp16 [z_0 .. z_{D/G-1}, s_0 .. s_{D/G-1}] (group g = elements
 * [gG, gG + G)).
 *
 * Conventions for every entry point:
 *   - All device buffers are allocated and owned by the caller.  The library
 *     allocates no device memory (kvq_decode_attention_static_ws uses a
 *     fixed array of its device image) and keeps no state between calls
 *     except host-side caches: the SM count per device, the kernel
 *     attributes it has set, and whether the runtime accepted programmatic
 *     dependent launch.
 *   - Every argument is checked on the host before any launch; a failed
 *     check returns a status and launches nothing.  A launch failure returns
 *     KVQ_ERR_CUDA.  Faults of already-launched kernels surface at the
 *     caller's next synchronisation.
 *   - Work is enqueued on `stream` (a cudaStream_t passed as void*; NULL is
 *     the legacy default stream) and never synchronised by the library.
 *   - The current CUDA device must be the one that owns the buffers.
 */
#ifndef KVQ_H_
#define KVQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KVQ_MAX_HEADS 128   /* H_kv limit (mask and slot tables are this long) */
#define KVQ_NSEG 8          /* number of cache segments */
#define KVQ_MAX_CTAS 1024   /* upper bound on split-KV work chunks per call */
#define KVQ_HEADS_PER_UNIT 8 /* query columns (query heads, or head x token pairs) handled together per KV head */
#define KVQ_MAX_QUERY_TOKENS 64 /* query tokens per sequence of kvq_decode_attention_mq */

/* Bits of the status word that the decode kernels OR into the first 4 bytes
 * of their workspace (never cleared by the library; zero it to start).  A
 * set bit means that some output rows of a call are NaN (or, for a corrupt
 * counter found by only some CTAs, unreliable):
 *   KVQ_STATUS_TILE_WAIT  a staged cache tile did not arrive within the
 *                         bounded wait (only a fault elsewhere causes it)
 *   KVQ_STATUS_PEER_WAIT  a combining CTA gave up waiting for the other
 *                         CTAs of its unit (their partials, in cluster
 *                         mode; the unit's last arrival, in the global-mode
 *                         kvq_decode_step(_ragged))
 *   KVQ_STATUS_COUNTER    an arrival counter of kvq_decode_step(_ragged) was
 *                         not zero when the call started (workspace not
 *                         zeroed, or shared by calls that overlap) */
#define KVQ_STATUS_TILE_WAIT 1u
#define KVQ_STATUS_PEER_WAIT 2u
#define KVQ_STATUS_COUNTER 4u

typedef enum kvq_status {
  KVQ_OK = 0,
  KVQ_ERR_INVALID_ARG = 1, /* null pointer, bad size, misaligned buffer, corrupt layout */
  KVQ_ERR_UNSUPPORTED = 2, /* valid but not implemented (e.g. D != 128) */
  KVQ_ERR_CAPACITY = 3,    /* positions beyond T_cap, or workspace too small */
  KVQ_ERR_CUDA = 4         /* a CUDA runtime call or kernel launch failed */
} kvq_status;

/* Segments of one layer's cache buffer (see kvq_layout.off / .bytes). */
enum kvq_segment {
  KVQ_SEG_K_CODES = 0, /* uint32 [B][n_packed][Tv_pad][D*k_bits/32] (storage order above); bf16 rows if k_bits == 16 */
  KVQ_SEG_K_SZ = 1,    /* fp16 [B][n_packed][Tv_pad][2*D/G] = [z.., s..]; empty if k_bits == 16 */
  KVQ_SEG_V_CODES = 2, /* as K_CODES with v_bits, [B][n_packed + n_konly][..]: packed heads, then K-only ones */
  KVQ_SEG_V_SZ = 3,    /* as K_SZ with v_bits, [B][n_packed + n_konly][..] */
  KVQ_SEG_PROT_K = 4,  /* bf16 [B][n_prot + n_konly][Tv][D]: visual K of protected, then K-only heads */
  KVQ_SEG_PROT_V = 5,  /* bf16 [B][n_prot][Tv][D]: visual V of protected heads */
  KVQ_SEG_TEXT_K = 6,  /* bf16 [B][H_kv][T_cap - Tv][D]: every non-visual position */
  KVQ_SEG_TEXT_V = 7   /* bf16 [B][H_kv][T_cap - Tv][D] */
};

/* Per-layer description of the cache (the pages' problem statement). */
typedef struct kvq_layout_desc {
  int32_t B;          /* sequences in the batch, >= 1 */
  int32_t H_q;        /* query heads, multiple of H_kv */
  int32_t H_kv;       /* KV heads, 1..KVQ_MAX_HEADS */
  int32_t D;          /* head dim; this build supports D == 128 */
  int32_t T_cap;      /* positions the cache can hold per sequence, >= 1 */
  int32_t vis_start;  /* visual range [vis_start, vis_end), 0 <= start <= end <= T_cap */
  int32_t vis_end;
  int32_t k_bits;     /* 2, 4, 8, or 16 (= bf16, unquantised) */
  int32_t v_bits;     /* 2, 4, 8, or 16 */
  int32_t group_size; /* G in {32, 64, 128}, groups of G consecutive elements along D */
  uint8_t protected_heads[KVQ_MAX_HEADS]; /* 0 = quantised; 1 = visual K and V of that KV head
                                             stay bf16; 2 = only its visual K stays bf16
                                             (HeadGuard's "K, and V as needed") */
} kvq_layout_desc;

/* Derived layout (plain value; filled by kvq_cache_layout, read-only after). */
typedef struct kvq_layout {
  kvq_layout_desc d;
  int32_t g;          /* H_q / H_kv */
  int32_t n_prot;     /* KV heads with K and V protected (mode 1) */
  int32_t n_packed;   /* unprotected KV heads */
  int32_t Tv;         /* vis_end - vis_start: visual rows per (b, head) */
  int32_t Tv_pad;     /* Tv rounded up to a multiple of 16: row stride of the packed segments */
  int32_t T_text;     /* T_cap - Tv: text rows per (b, head) */
  int32_t units;      /* B * H_kv * ceil(g / KVQ_HEADS_PER_UNIT) */
  int32_t slot[KVQ_MAX_HEADS];        /* head -> index among its kind (protected / K-only / packed) */
  uint8_t prot_head[KVQ_MAX_HEADS];   /* protected slot -> head */
  uint8_t packed_head[KVQ_MAX_HEADS]; /* packed slot -> head (mode 0) */
  int64_t row_bytes[KVQ_NSEG];        /* bytes of one row of each segment */
  int64_t off[KVQ_NSEG];              /* byte offset of each segment (256-byte aligned) */
  int64_t bytes[KVQ_NSEG];            /* payload bytes of each segment */
  int64_t total_bytes;                /* size of the cache buffer (segments + padding) */
  int64_t workspace_bytes;            /* decode workspace needed for any T <= T_cap */
  double eff_bits_k;                  /* stored bits per visual K value, scale/zero included */
  double eff_bits_v;
  int32_t n_konly;                    /* KV heads with only K protected (mode 2) */
  uint8_t konly_head[KVQ_MAX_HEADS];  /* K-only slot -> head */
} kvq_layout;

/*
 * kvq_cache_layout -- host only, pure.  Validates `desc` and fills `out`:
 * which head goes to which segment slot, segment offsets and sizes, the
 * effective bits per value (b + 32/G for quantised tensors, 16 otherwise)
 * and the decode workspace size.  Returns KVQ_ERR_INVALID_ARG for a null
 * pointer or an inconsistent description, KVQ_ERR_UNSUPPORTED for D != 128.
 */
kvq_status kvq_cache_layout(const kvq_layout_desc* desc, kvq_layout* out);

/*
 * kvq_quantize_append -- write positions [t0, t0 + n_tok) of every sequence
 * into the cache ("VLM_KV_Quantization" section 1: historical visual K/V at
 * INT8/INT4/INT2 with a group size; HeadGuard: protected heads stay bf16).
 *   L        layout from kvq_cache_layout (host pointer, copied by value)
 *   cache    device buffer of L->total_bytes, 256-byte aligned
 *   k_bf16, v_bf16   device bf16 tensors [B][H_kv][n_tok][D]; element
 *            (b, h, i, d) at index b*stride_b + h*stride_h + i*stride_t + d
 *            (strides in elements, multiples of 8; d contiguous; tensors
 *            16-byte aligned)
 *   t0, n_tok  first position and count; n_tok == 0 is a no-op
 * A position in [vis_start, vis_end) of an unprotected head is quantised
 * (bits < 16) and packed; every other position is copied bf16 verbatim.
 * Returns KVQ_ERR_CAPACITY if t0 + n_tok > T_cap.
 */
kvq_status kvq_quantize_append(const kvq_layout* L, void* cache, const void* k_bf16,
                               const void* v_bf16, int64_t stride_b, int64_t stride_h,
                               int64_t stride_t, int32_t t0, int32_t n_tok, void* stream);

/*
 * kvq_decode_attention -- one decode query per sequence attends to positions
 * [0, T) of the cache (split-KV flash decoding; dequantisation happens in
 * registers and no dequantised K/V is ever written to device memory).
 *   q_bf16    device bf16 [B][H_q][D], 16-byte aligned
 *   T         attended positions, 1 <= T <= T_cap (all appended before)
 *   softmax_scale  multiplies q.k (e.g. 1/sqrt(D))
 *   out_bf16  device bf16 [B][H_q][D], 16-byte aligned
 *   lse       device fp32 [B][H_q] (natural-log sum of exp of the scaled
 *             scores) or NULL
 *   workspace device scratch of at least L->workspace_bytes, 256-byte
 *             aligned; its first 4 bytes are the status word (KVQ_STATUS_*
 *             bits OR-ed in by the kernels, never cleared by the library:
 *             zero it to use it, read it with kvq_workspace_status); other
 *             contents on entry are ignored; overlapping calls must not
 *             share one workspace
 * out[b, hq, :] = sum_p softmax_p(scale * q[b,hq] . khat[b,h,p]) * vhat[b,h,p],
 * h = hq / g, where khat/vhat are the dequantised (or bf16) cache rows.
 * Returns KVQ_ERR_CAPACITY if ws_bytes < L->workspace_bytes.
 */
kvq_status kvq_decode_attention(const kvq_layout* L, const void* cache, const void* q_bf16,
                                int32_t T, float softmax_scale, void* out_bf16, float* lse,
                                void* workspace, size_t ws_bytes, void* stream);

/*
 * kvq_decode_step -- one decode step of one layer in a single launch: the
 * step's own K/V row is written into the cache at text position t_new
 * (never quantised: "VLM_KV_Quantization", intro checklist) and the step's
 * query attends to positions [0, t_new] (WSVD summary, section 2.라 flash
 * decoding with on-chip reconstruction).  Same result as
 * kvq_quantize_append(t0 = t_new, n_tok = 1) followed by
 * kvq_decode_attention(T = t_new + 1), up to the summation order of the
 * cross-split combine.  The append, the split-KV pass and the combine run in
 * one kernel, in one of two ways chosen per call:
 *   - cluster mode, when every (b, KV head, query-head chunk) unit fits one
 *     16-CTA thread-block cluster resident on the GPU and a sixteenth of a
 *     unit is small: each CTA of a unit's cluster stores its partial of
 *     column j into the shared memory of the cluster's CTA j (asynchronous
 *     distributed-shared-memory stores counted on that CTA's barrier),
 *     which waits (bounded) for them and writes the row; no CTA waits for
 *     another cluster;
 *   - global mode otherwise: CTAs publish partials in the workspace and
 *     count arrivals on a per-unit counter; the last min(chunks, heads)
 *     arrivals of a unit combine its rows, the earlier of them waiting
 *     (bounded) until the very last arrival has reset the counter, so the
 *     launch is cooperative (all CTAs resident).
 *   k_new_bf16, v_new_bf16  device bf16 [B][H_kv][D], contiguous, 16-byte aligned
 *   t_new      0 <= t_new < T_cap, outside [vis_start, vis_end)
 *   workspace  as for kvq_decode_attention; in addition, after its
 *              256-byte head (status word), the next
 *              ceil(4 * L->units / 256) * 256 bytes hold the arrival
 *              counters and must be zero before the first kvq_decode_step
 *              call that uses the workspace (zero the whole workspace once
 *              after allocating it).  Every call leaves them zero again.
 *              Other workspace bytes are ignored on entry.  Calls sharing
 *              one workspace must be ordered (one stream), and use layouts
 *              with the same L->units (the counter area's size), or zero
 *              the workspace again when switching.
 * A bounded wait that gives up (a staged tile that does not arrive, or in
 * global mode a combining CTA whose unit's last arrival does not come) and
 * an arrival counter found non-zero at entry never hang the call: the
 * affected output rows become NaN and the KVQ_STATUS_* bit is OR-ed into
 * the workspace status word.
 */
kvq_status kvq_decode_step(const kvq_layout* L, void* cache, const void* q_bf16,
                           const void* k_new_bf16, const void* v_new_bf16, int32_t t_new,
                           float softmax_scale, void* out_bf16, float* lse, void* workspace,
                           size_t ws_bytes, void* stream);

/*
 * Ragged batches: every sequence of the batch has its own length, held in a
 * device array that the caller's decode loop updates on the GPU (so the
 * calls can be captured once in a CUDA graph and replayed as lengths grow).
 * The layout (visual range, protected heads) is shared by the batch; a
 * sequence attends only to its own positions.  Work is split over T_max
 * positions per sequence, so the cost is that of a uniform call of length
 * T_max whatever the lengths are.
 *
 * kvq_decode_attention_ragged -- kvq_decode_attention with sequence b
 * attending positions [0, seq_len[b]).
 *   seq_len   device int32 [B], 4-byte aligned, read by the kernels (after
 *             the previous kernel of the stream has finished)
 *   T_max     1 <= T_max <= T_cap; entries are meant to lie in [1, T_max]
 * An entry outside [1, T_max] marks an inactive sequence: its outputs are
 * zero and its lse is -inf (no error is returned; the host never sees the
 * array).  The other arguments are those of kvq_decode_attention.
 */
kvq_status kvq_decode_attention_ragged(const kvq_layout* L, const void* cache, const void* q_bf16,
                                       const int32_t* seq_len, int32_t T_max, float softmax_scale,
                                       void* out_bf16, float* lse, void* workspace, size_t ws_bytes,
                                       void* stream);

/*
 * kvq_decode_step_ragged -- kvq_decode_step with one step position per
 * sequence: sequence b stores its K/V row at t_new[b] and attends positions
 * [0, t_new[b]].
 *   t_new     device int32 [B], 4-byte aligned
 *   T_max     1 <= T_max <= T_cap; entries are meant to lie in [0, T_max)
 *             and outside [vis_start, vis_end)
 * An entry outside that set marks an inactive sequence: nothing is stored
 * for it, its outputs are zero and its lse is -inf.  The workspace rules
 * are those of kvq_decode_step (the arrival counters are shared by both
 * step entry points).
 */
kvq_status kvq_decode_step_ragged(const kvq_layout* L, void* cache, const void* q_bf16,
                                  const void* k_new_bf16, const void* v_new_bf16,
                                  const int32_t* t_new, int32_t T_max, float softmax_scale,
                                  void* out_bf16, float* lse, void* workspace, size_t ws_bytes,
                                  void* stream);

/*
 * kvq_decode_attention_mq -- multi-query decode: n_q query tokens per
 * sequence (draft tokens being verified, or a chunk of new tokens), whose
 * own K/V rows were appended at positions [T - n_q, T) before the call.
 * Token i attends positions [0, T - n_q + 1 + i) (causal among the new
 * tokens).  The (query head, token) pairs of a KV head share one pass over
 * its cache: up to KVQ_HEADS_PER_UNIT of them are the N = 8 columns of one
 * tensor-core tile (WSVD summary, section 2.라: QK, softmax and PV fused),
 * so an MHA layer (g = 1) fills the tile with 8 tokens.
 *   q_bf16    device bf16 [B][n_q][H_q][D], 16-byte aligned
 *   n_q       1 <= n_q <= KVQ_MAX_QUERY_TOKENS
 *   T         n_q <= T <= T_cap; the positions some token does not attend,
 *             [T - n_q + 1, T), must lie outside [vis_start, vis_end)
 *   out_bf16  device bf16 [B][n_q][H_q][D];  lse  fp32 [B][n_q][H_q] or NULL
 *   workspace at least kvq_decode_mq_workspace_bytes(L, n_q) bytes (equal to
 *             L->workspace_bytes for n_q = 1), 256-byte aligned
 * n_q = 1 is kvq_decode_attention.  Other arguments and errors as there.
 * kvq_decode_mq_workspace_bytes returns 0 for an invalid layout or n_q
 * outside [1, KVQ_MAX_QUERY_TOKENS].
 */
size_t kvq_decode_mq_workspace_bytes(const kvq_layout* L, int32_t n_q);
kvq_status kvq_decode_attention_mq(const kvq_layout* L, const void* cache, const void* q_bf16,
                                   int32_t n_q, int32_t T, float softmax_scale, void* out_bf16,
                                   float* lse, void* workspace, size_t ws_bytes, void* stream);

/*
 * kvq_sensitivity_probe -- how far the cache's quantisation moves attention,
 * the model-free form of the K-vs-V study of "VLM_KV_Quantization",
 * sections 3-4 (KL divergence of the distribution after quantising visual
 * K or visual V alone -- same tokens, bits and group size -- from the
 * unquantised one).  For every (b, hq), h = hq / g, in fp64:
 *   kl_attn = D_KL(p || p_hat): p = softmax_t(scale q.k_t) over the raw bf16
 *             K rows, p_hat the same over K as kvq_decode_attention reads it
 *             (dequantised code * s + z, or the bf16 side store);
 *   kl_out  = D_KL(P || P_hat): P = softmax(readout o), o the attention
 *             output over the raw K/V rows, P_hat the same over the cache;
 *   err     = ||o_hat - o||_2.
 * To compare K with V, run it on two caches appended from the same rows with
 * layouts that differ only in k_bits / v_bits (16 = unquantised).
 *   cache, q_bf16, T, softmax_scale  as for kvq_decode_attention (positions [0, T))
 *   k_bf16, v_bf16  device bf16, the raw rows that were appended: element
 *             (b, h, t, d) at index b*stride_b + h*stride_h + t*stride_t + d;
 *             16-byte aligned, strides >= 0 and multiples of 8 elements
 *   readout   device fp32 [n_out][D], 8-byte aligned, 1 <= n_out <= 2048
 *   result    device fp64 [B][H_q][3] = (kl_attn, kl_out, err), 8-byte aligned
 *   workspace device scratch of at least kvq_probe_workspace_bytes(L, T)
 *             bytes, 16-byte aligned; contents on entry are ignored
 * Returns KVQ_ERR_UNSUPPORTED for D != 128 or B * H_q > 65535.
 * kvq_probe_workspace_bytes returns 0 for an invalid layout or T < 1.
 */
size_t kvq_probe_workspace_bytes(const kvq_layout* L, int32_t T);
kvq_status kvq_sensitivity_probe(const kvq_layout* L, const void* cache, const void* q_bf16,
                                 const void* k_bf16, const void* v_bf16, int64_t stride_b,
                                 int64_t stride_h, int64_t stride_t, int32_t T, float softmax_scale,
                                 const float* readout, int32_t n_out, double* result, void* workspace,
                                 size_t ws_bytes, void* stream);

/* Size in bytes of the device scratch array used by
 * kvq_decode_attention_static_ws (16 MiB).  A layout fits when
 * L->workspace_bytes <= KVQ_STATIC_WS_BYTES, which holds for up to 3007
 * units (B * H_kv * ceil(g/8) <= 3007). */
#define KVQ_STATIC_WS_BYTES (16u * 1024u * 1024u)

/*
 * kvq_decode_attention_static_ws -- the pages have no counterpart to this
 * entry point; it exists for callers that are not allowed to allocate
 * device memory (for example a plug-in whose host framework owns every
 * device allocation, or a serving loop that must never allocate).
 * It computes exactly what kvq_decode_attention computes, with the same
 * arguments minus the workspace: the split-KV scratch lives in a fixed
 * KVQ_STATIC_WS_BYTES array inside the library's device image, present on
 * every GPU that loads the library until the process exits.  No device
 * memory is allocated by this call.
 *   - Returns KVQ_ERR_CAPACITY, before any CUDA call, when
 *     L->workspace_bytes > KVQ_STATIC_WS_BYTES.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, once per device); make that first call before
 *     any stream capture on that device.
 *   - All calls on a device share the one array.  Calls whose kernels may
 *     run at the same time on the GPU (unordered streams) race on it; order
 *     them on one stream or use kvq_decode_attention with separate
 *     workspaces.  The array's contents on entry do not matter.
 */
kvq_status kvq_decode_attention_static_ws(const kvq_layout* L, const void* cache,
                                          const void* q_bf16, int32_t T, float softmax_scale,
                                          void* out_bf16, float* lse, void* stream);

/*
 * kvq_workspace_status -- enqueue on `stream` a copy of the workspace's
 * status word (KVQ_STATUS_* bits of every call that used the workspace
 * since it was last zeroed) into *status (host memory; pinned memory keeps
 * the copy asynchronous).  The value is there once the stream has reached
 * this point (synchronise it).  KVQ_ERR_INVALID_ARG for null or misaligned
 * pointers, KVQ_ERR_CUDA if the copy cannot be enqueued.
 */
kvq_status kvq_workspace_status(const void* workspace, uint32_t* status, void* stream);

/*
 * kvq_set_wait_limits -- for decode calls made later from the calling host
 * thread: how many times a kernel polls a staged tile's barrier
 * (tile_polls; each poll suspends the thread for a hardware-chosen
 * interval) and, in the global-mode fused step, the unit's counter
 * (peer_polls; each poll followed by a ~32 ns sleep) before the wait gives
 * up.  0 restores the default (2^24 and 2^21).  The defaults are far beyond
 * any healthy wait; shorter limits exist for testing the failure path.
 */
void kvq_set_wait_limits(uint32_t tile_polls, uint32_t peer_polls);

/*
 * kvq_set_cache_preload -- for decode calls made later from the calling host
 * thread: with enable != 0, the uniform single-query calls
 * (kvq_decode_attention, kvq_decode_attention_static_ws,
 * kvq_decode_attention_mq with n_q = 1, kvq_decode_step) that run in
 * cluster mode (see kvq_decode_step: every unit's share of a CTA fits its
 * shared-memory ring) copy each CTA's first cache tiles into shared memory
 * before the previous kernel in the stream has finished (programmatic
 * dependent launch), so a chain of layers overlaps one layer's cache reads
 * with the previous layer's work.  Only cache rows are read early; q, k_new
 * and v_new after the wait.
 *
 * Requirement: every kernel that writes the cache before the call in its
 * stream is a call of this library, or the host synchronises with it (or
 * a memory copy separates it) before the call.  The library's own writers
 * (kvq_quantize_append, kvq_decode_step, kvq_decode_step_ragged) fence
 * their cache writes and let the next kernel launch only after them and
 * after their own dependency wait, which makes the early copies see every
 * row written before.  Off (0) by default.
 */
void kvq_set_cache_preload(int32_t enable);

/* The cudaError_t value (as int) of the last CUDA call that made an entry
 * point return KVQ_ERR_CUDA on the calling host thread; 0 if none. */
int kvq_last_cuda_error(void);

/* Human-readable name of a status code (static string). */
const char* kvq_status_string(kvq_status s);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H_ */
