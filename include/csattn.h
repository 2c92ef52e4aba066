/*
 * csattn -- causal multi-head scaled dot-product attention with RoPE and
 * grouped-query KV heads, for one NVIDIA GB300 (sm_103a).
 *
 * The operation, as the source pages state it:
 *   Attn(Q,K,V;M) = softmax(Q K^T * scale + M) V, computed per head
 *     ("Transformer" (ai-notes), section "Scaled dot-product attention";
 *      "The Transformer architecture" (cooking-agi), same section, which also
 *      fixes the default scale 1/sqrt(d_head) of each head);
 *   M[t,s] = 0 for s <= t and -inf for s > t (causal)
 *     ("Transformer" (ai-notes), section "What is the causal mask?";
 *      "Transformer Math and Implementation Deep Dive", section "Causal Masking");
 *   q [B, n_q_heads, T, d_head], k and v [B, n_kv_heads, T, d_head], with
 *   n_q_heads a multiple of n_kv_heads and query head h reading KV head
 *   h / (n_q_heads / n_kv_heads)
 *     ("Transformer Math and Implementation Deep Dive", section "Attention Shapes");
 *   RoPE on q and k only, pair p of channels turned by pos * base^(-2p/d)
 *     ("The Transformer architecture", section "Now: RoPE" for the split-half
 *      pairing; "Transformer" (ai-notes), section "RoPE (Rotary Positional
 *      Embedding)" for the adjacent pairing and the angle formula);
 *   KV-cache decode: the new query at position L-1 sees cached rows 0..L-1
 *     ("The Transformer architecture", section "Hands-on").
 *
 * Conventions for every call:
 *   - All tensors are dense, row-major, contiguous, in device memory, and
 *     16-byte aligned (they are read by TMA).  The caller owns every buffer;
 *     the library allocates no device memory at run time: its only device
 *     memory is static (one status word per device, and the scratch buffer
 *     of csattn_attn_decode_noalloc).
 *   - Calls are asynchronous on `stream` (a cudaStream_t, NULL = legacy default
 *     stream) and never synchronize.  Argument errors are detected on the host
 *     before any launch and returned; nothing is launched then.
 *   - Kernels never trap.  A wait that runs out of time (a hang) or a failed
 *     device-side check raises a bit in the device status word;
 *     csattn_check_status() reads and clears it.
 *   - Return value: a csattn_status; csattn_last_error() gives a message for
 *     the last failure on the calling thread.
 */
#ifndef CSATTN_H_
#define CSATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  CSATTN_OK = 0,
  CSATTN_ERR_INVALID_ARG = -1,  /* bad shape, pointer, alignment or value      */
  CSATTN_ERR_UNSUPPORTED = -2,  /* valid but not implemented (d, dtype, group) */
  CSATTN_ERR_CUDA = -3,         /* a CUDA runtime/driver call failed           */
  CSATTN_ERR_TIMEOUT = -4,      /* a kernel wait ran out of time (status word) */
  CSATTN_ERR_WORKSPACE = -5,    /* workspace missing or too small              */
  CSATTN_ERR_DEVICE_ARG = -6    /* a device-side check failed (status word)    */
} csattn_status;

typedef enum { CSATTN_F32 = 0, CSATTN_BF16 = 1 } csattn_dtype;

typedef enum { CSATTN_ROPE_SPLIT_HALF = 0, CSATTN_ROPE_ADJACENT = 1 } csattn_rope_layout;

/* OR into rope_layout of csattn_attn_fwd: k is already rotated (for instance
 * by csattn_rope_rotate, as a KV cache stores it); only q is rotated. */
#define CSATTN_ROPE_K_PREROTATED 0x100

/*
 * Bytes of device workspace csattn_attn_fwd needs for these arguments.
 * Non-zero only for bf16 with RoPE (rope_base > 0): the rotated keys,
 * B*Hkv*T*d bf16 values, which are computed once per call rather than once
 * per query tile.  Returns 0 as well for arguments that csattn_attn_fwd
 * would reject.
 */
size_t csattn_fwd_workspace_size(int B, int Hq, int Hkv, int T, int d, int dtype,
                                 float rope_base);

/*
 * Prefill forward: out = softmax(RoPE(q) RoPE(k)^T * scale + M) v.
 *   q    [B, Hq,  T, d]   dtype `dtype` (CSATTN_BF16 or CSATTN_F32)
 *   k, v [B, Hkv, T, d]   same dtype
 *   out  [B, Hq,  T, d]   same dtype, written (rounded to nearest even)
 *   causal       1: M is the causal mask; 0: no mask (M = 0).
 *   rope_base    > 0: RoPE with theta_p = rope_base^(-2p/d) at positions
 *                0..T-1 on q and k; <= 0: no RoPE.
 *   rope_layout  CSATTN_ROPE_SPLIT_HALF (channel p with p + d/2) or
 *                CSATTN_ROPE_ADJACENT (channel 2p with 2p+1), optionally OR
 *                CSATTN_ROPE_K_PREROTATED (k given rotated; no workspace needed).
 *   scale        > 0: logit scale; <= 0: 1/sqrt(d).
 *   lse          NULL, or fp32 [B, Hq, T]: natural-log log-sum-exp of each
 *                scaled, masked score row.
 *   workspace    device buffer of at least csattn_fwd_workspace_size() bytes
 *                (may be NULL when that size is 0), owned by the caller.
 * Requirements: B, Hq, Hkv, T >= 1; Hq % Hkv == 0; d in {64, 128} for bf16,
 * d in {16, 32, 64, 128} for fp32; T < 2^24, and T <= 49152 with RoPE (the
 * range in which the angles are reduced exactly).  The rotated q and k are rounded
 * to the input dtype before the dot products; accumulation is fp32.
 */
int csattn_attn_fwd(const void* q, const void* k, const void* v, void* out, int B, int Hq,
                    int Hkv, int T, int d, int dtype, int causal, float rope_base,
                    int rope_layout, float scale, float* lse, void* workspace,
                    size_t workspace_bytes, void* stream);

/*
 * Bytes of device workspace csattn_attn_fwd_host needs: device copies of q, k, v,
 * out and lse, and the rotated keys (each block 256-byte aligned).  0 for an
 * unknown dtype or a size below 1.
 */
size_t csattn_fwd_host_workspace_size(int B, int Hq, int Hkv, int T, int d, int dtype,
                                      float rope_base);

/*
 * csattn_attn_fwd on HOST buffers: q, k, v are read from host memory and out (and
 * lse, if non-NULL) written to host memory, all in the layouts of csattn_attn_fwd.
 * The problem is cut into num_chunks chunks of consecutive (sequence, KV head)
 * pairs (a pair owns its Hq / Hkv query heads, so a chunk is contiguous in every
 * tensor); each chunk's inputs are copied in, its attention computed and its output
 * copied out on three internal streams of the current device, so that the copies of
 * one chunk overlap the kernels and the opposite-direction copies of the others.
 * The results equal csattn_attn_fwd's bit for bit.
 *   q_h, k_h, v_h, out_h, lse_h  host pointers; page-locked memory (cudaHostAlloc or
 *                cudaHostRegister) lets the copies run asynchronously
 *   num_chunks   0: automatic (16, at most B * Hkv); otherwise 1..16 (capped at B*Hkv)
 *   workspace    device buffer of >= csattn_fwd_host_workspace_size() bytes,
 *                16-byte aligned, in use until the call's work on `stream` completes
 * Other arguments, checks and return codes as csattn_attn_fwd (messages name
 * attn_fwd_host).  Every check runs before the first copy is enqueued.  Asynchronous
 * on `stream`: the internal streams wait for the work already on `stream`, and
 * `stream` waits for the last copy out; the host buffers must stay valid until then
 * (also after an error returned once copies were enqueued: `stream` then waits for
 * everything already enqueued).  Concurrent calls from several host threads are
 * serialised while they enqueue.
 */
int csattn_attn_fwd_host(const void* q_h, const void* k_h, const void* v_h, void* out_h, int B,
                         int Hq, int Hkv, int T, int d, int dtype, int causal, float rope_base,
                         int rope_layout, float scale, float* lse_h, int num_chunks,
                         void* workspace, size_t workspace_bytes, void* stream);

/*
 * Bytes of device workspace csattn_attn_fwd_ext needs: the rotated keys,
 * B*Hkv*Tk*d*2, for bf16 with RoPE (unless k is given rotated); 0 otherwise.
 */
size_t csattn_fwd_ext_workspace_size(int B, int Hq, int Hkv, int Tq, int Tk, int d, int dtype,
                                     float rope_base);

/*
 * Prefill of a chunk of queries after a cache prefix, or rectangular
 * (cross-)attention ("The Transformer architecture", "Hands-on": the query at
 * position p sees cached keys 0..p; "Transformer Math and Implementation Deep
 * Dive", "Attention Equation": Tq and Tk need not match without a mask).
 *   q    [B, Hq,  Tq, d];  k [B, Hkv, Tk, d];  v [B, Hkv, Tk, dv];  out [B, Hq, Tq, dv]
 *   dv           head size of v and out ("Scaled dot-product attention": the
 *                values need not have the keys' width); <= 0 means dv = d.
 *                bf16: d, dv in {64, 128}; fp32: d, dv in {16, 32, 64, 128}.
 *                The default scale stays 1/sqrt(d) and RoPE acts on q and k.
 *   q_offset     position of query row 0: row i sits at q_offset + i; keys sit
 *                at 0..Tk-1.  With causal = 1, row i sees keys j <= q_offset + i
 *                (a chunked prefill passes Tk = q_offset + Tq: the cached prefix
 *                followed by the chunk's own keys).  With causal = 0 every key
 *                is visible.
 *   rope_base    > 0: q is rotated at positions q_offset + i and k at 0..Tk-1
 *                (unless CSATTN_ROPE_K_PREROTATED is set in rope_layout).
 *   lse          NULL or fp32 [B, Hq, Tq].
 *   workspace    at least csattn_fwd_ext_workspace_size() bytes.
 * Other arguments, ownership and errors as csattn_attn_fwd, which is this call
 * with Tq = Tk = T and q_offset = 0.  Additional requirements: Tq, Tk >= 1,
 * 0 <= q_offset < 2^24; with RoPE, q_offset + Tq <= 49152 and Tk <= 49152
 * (CSATTN_ERR_UNSUPPORTED otherwise).
 */
int csattn_attn_fwd_ext(const void* q, const void* k, const void* v, void* out, int B, int Hq,
                        int Hkv, int Tq, int Tk, int q_offset, int d, int dv, int dtype,
                        int causal, float rope_base, int rope_layout, float scale, float* lse,
                        void* workspace, size_t workspace_bytes, void* stream);

/*
 * Bytes of device workspace csattn_attn_bwd needs: fp32 rowsum(dout o out)
 * [B, Hq, T] plus, with RoPE, the rotated q and k in the input dtype (each
 * block 256-byte aligned).  0 for an unknown dtype or a size below 1.
 */
size_t csattn_bwd_workspace_size(int B, int Hq, int Hkv, int T, int d, int dtype,
                                 float rope_base);

/*
 * Backward of csattn_attn_fwd: the gradients of sum(out * dout) with respect to
 * q, k and v.  Written out from the forward's definition ("The Transformer
 * architecture", "Scaled dot-product attention", "Now: RoPE"):
 *   P = exp(S - lse), S = scale * RoPE(q) RoPE(k)^T + M;  D = rowsum(dout o out)
 *   dv = sum over the group's query heads of P^T dout
 *   dS = P o (dout v^T - D)
 *   dq = R^T (scale * dS RoPE(k)),  dk = R^T (scale * sum over heads of dS^T RoPE(q))
 * with R the rotation at each row's position (R^T = R^-1).  The rounding of the
 * rotated operands in the forward is taken as the identity.
 *   q, k, v, causal, rope_base, rope_layout, scale   the forward's arguments
 *   out   [B, Hq, T, d]  the forward's output;  dout [B, Hq, T, d] its gradient
 *   lse   fp32 [B, Hq, T] the forward's natural-log log-sum-exp (its lse output)
 *   dq [B, Hq, T, d], dk, dv [B, Hkv, T, d]  written, same dtype as q
 *   workspace  >= csattn_bwd_workspace_size() bytes, caller-owned
 * Requirements: bf16 with d in {64, 128} (tcgen05 kernels) or fp32 with d in
 * {16, 32, 64, 128} (SIMT kernels, fp32 throughout, RoPE with the accurate
 * sine/cosine); other d CSATTN_ERR_UNSUPPORTED.  Hq % Hkv == 0, T < 2^24
 * (T <= 49152 with RoPE); all pointers 16-byte aligned (lse 4-byte).
 * Asynchronous on `stream`.
 */
int csattn_attn_bwd(const void* q, const void* k, const void* v, const void* out,
                    const void* dout, const float* lse, void* dq, void* dk, void* dv, int B,
                    int Hq, int Hkv, int T, int d, int dtype, int causal, float rope_base,
                    int rope_layout, float scale, void* workspace, size_t workspace_bytes,
                    void* stream);

/*
 * Bytes of device workspace csattn_attn_bwd_ext needs: fp32 rowsum(dout o out)
 * [B, Hq, Tq] plus, with RoPE, the rotated q [B, Hq, Tq, d] and k [B, Hkv, Tk, d]
 * in the input dtype (each block 256-byte aligned).  0 for an unknown dtype or a
 * size below 1.
 */
size_t csattn_bwd_ext_workspace_size(int B, int Hq, int Hkv, int Tq, int Tk, int d, int dtype,
                                     float rope_base);

/*
 * Backward of csattn_attn_fwd_ext: the gradients of sum(out * dout) for a chunk
 * of Tq queries after a prefix ("The Transformer architecture", "Hands-on": the
 * query at position p sees keys 0..p) or for rectangular attention, with value
 * width d_v ("Transformer Math and Implementation Deep Dive", "Attention
 * Equation": Tq and Tk, d_k and d_v need not match).  The formulas are those of
 * csattn_attn_bwd with the mask and positions of csattn_attn_fwd_ext: query row i
 * sits at position q_offset + i, key j at j; with causal = 1 row i sees keys
 * j <= q_offset + i, with causal = 0 every key.
 *   q [B, Hq, Tq, d];  k [B, Hkv, Tk, d];  v [B, Hkv, Tk, d_v]
 *   out, dout    [B, Hq, Tq, d_v]: the forward's output and its gradient
 *   lse          fp32 [B, Hq, Tq]: the forward's natural-log log-sum-exp
 *   dq [B, Hq, Tq, d], dk [B, Hkv, Tk, d], dv [B, Hkv, Tk, d_v]  written, q's dtype.
 *                A key no query sees (causal, j > q_offset + Tq - 1) gets dk = dv = 0.
 *   d_v          <= 0 means d_v = d.  bf16: d, d_v in {64, 128} (tcgen05 kernels);
 *                fp32: d, d_v in {16, 32, 64, 128} (SIMT kernels, fp32 throughout).
 *   rope_base    > 0: q is rotated at q_offset + i and k at 0..Tk-1 (both given
 *                unrotated: CSATTN_ROPE_K_PREROTATED is CSATTN_ERR_UNSUPPORTED);
 *                dq and dk are the gradients with respect to the unrotated q and k.
 *   workspace    >= csattn_bwd_ext_workspace_size() bytes, 16-byte aligned,
 *                caller-owned, in use until the call's work on `stream` completes.
 * Other arguments, ownership and errors as csattn_attn_bwd, which is this call
 * with Tq = Tk = T, q_offset = 0 and d_v = d.  Requirements: Tq, Tk >= 1,
 * 0 <= q_offset < 2^24, Tq, Tk < 2^24; with RoPE q_offset + Tq <= 49152 and
 * Tk <= 49152 (CSATTN_ERR_UNSUPPORTED otherwise).  Asynchronous on `stream`.
 */
int csattn_attn_bwd_ext(const void* q, const void* k, const void* v, const void* out,
                        const void* dout, const float* lse, void* dq, void* dk, void* dv, int B,
                        int Hq, int Hkv, int Tq, int Tk, int q_offset, int d, int d_v, int dtype,
                        int causal, float rope_base, int rope_layout, float scale,
                        void* workspace, size_t workspace_bytes, void* stream);

/*
 * RoPE of x [B, H, T, d] into x_rot (same shape; must not overlap x), at
 * positions 0..T-1 with theta_p = rope_base^(-2p/d), rounded to the input
 * dtype.  This is the rotation csattn_attn_fwd applies to its keys, exposed to
 * build a rotated KV cache for csattn_attn_decode.  bf16 with d in {64, 128}, or
 * fp32 with d in {16, 32, 64, 128} (fp32 arithmetic, the accurate sine/cosine, as
 * the fp32 prefill rotates); rope_base > 0; T <= 49152.
 */
int csattn_rope_rotate(const void* x, void* x_rot, int B, int H, int T, int d, int dtype,
                       float rope_base, int rope_layout, void* stream);

/*
 * Bytes of device workspace csattn_attn_decode needs: fp32 partial results
 * (running max, sum and un-normalised output) of every key split.
 * num_splits = 0 means the automatic choice (the size then covers any
 * max_seq_len <= Lmax); otherwise the explicit number of splits.
 */
size_t csattn_decode_workspace_size(int B, int Hq, int Lmax, int d, int num_splits);

/*
 * KV-cache decode: one new query per sequence.
 *   q        [B, Hq, 1, d]     already rotated to position seq_lens[b]-1
 *   k_cache  [B, Hkv, Lmax, d] keys already rotated (RoPE) at their positions
 *   v_cache  [B, Hkv, Lmax, d]
 *   seq_lens device int32 [B]: valid rows of sequence b, 1 <= seq_lens[b] <= max_seq_len
 *   out      [B, Hq, 1, d]
 *   dtype    CSATTN_BF16 (d in {64, 128}, Hq / Hkv <= 16; tensor-core kernels) or
 *            CSATTN_F32 (d in {16, 32, 64, 128}; SIMT kernels in fp32 throughout, for
 *            callers that want the decode close to float64), all tensors that dtype
 *   scale    > 0: logit scale; <= 0: 1/sqrt(d)
 *   max_seq_len  host-side upper bound of seq_lens (<= Lmax); sizes the grid.
 *   num_splits   0: automatic; > 0: split every sequence's keys into that many
 *                parts (a testing and tuning knob; results agree to rounding).
 *   workspace    >= csattn_decode_workspace_size(B, Hq, Lmax, d, num_splits) bytes.
 * Rows at or beyond seq_lens[b] are never read.  A seq_lens[b] outside
 * [1, max_seq_len] raises CSATTN_ERR_DEVICE_ARG in the status word (the
 * sequence's output is then zero or partial).  Requirements: Hq % Hkv == 0 and
 * the dtype's d (and group size) above; the other decode calls are bf16 only.
 */
int csattn_attn_decode(const void* q, const void* k_cache, const void* v_cache,
                       const int32_t* seq_lens, void* out, int B, int Hq, int Hkv, int Lmax,
                       int d, int dtype, float scale, int max_seq_len, int num_splits,
                       void* workspace, size_t workspace_bytes, void* stream);

/*
 * csattn_attn_decode with values of their own width dv ("Transformer Math and
 * Implementation Deep Dive", "Attention Equation": the weights come from q and k,
 * v sets the output width).
 *   q [B, Hq, 1, d];  k_cache [B, Hkv, Lmax, d];  v_cache [B, Hkv, Lmax, dv];
 *   out [B, Hq, 1, dv]
 *   d, dv        each 64 or 128 (CSATTN_ERR_UNSUPPORTED otherwise); dv <= 0 means
 *                dv = d, which is csattn_attn_decode.  The default scale is 1/sqrt(d).
 *   workspace    >= csattn_decode_workspace_size(B, Hq, Lmax, dv, num_splits) bytes
 *                (the split partials have the width of v).
 * Other arguments, checks and errors as csattn_attn_decode (messages name
 * attn_decode_ext).
 */
int csattn_attn_decode_ext(const void* q, const void* k_cache, const void* v_cache,
                           const int32_t* seq_lens, void* out, int B, int Hq, int Hkv, int Lmax,
                           int d, int dv, int dtype, float scale, int max_seq_len,
                           int num_splits, void* workspace, size_t workspace_bytes,
                           void* stream);

/*
 * Bytes of device workspace csattn_attn_decode_host needs: device copies of q, the
 * two caches (full [B, Hkv, Lmax, d] layout, only the visible rows written), the
 * lengths and out, and the split partials of csattn_decode_workspace_size().
 */
size_t csattn_decode_host_workspace_size(int B, int Hq, int Hkv, int Lmax, int d,
                                         int num_splits);

/*
 * csattn_attn_decode on HOST buffers: q [B, Hq, 1, d], the caches [B, Hkv, Lmax, d]
 * and seq_lens [B] (int32) in host memory, out [B, Hq, 1, d] written to host memory.
 * Only the rows the decode reads cross the host link: rows 0..seq_lens[b]-1 of every
 * KV head of sequence b (one strided copy per sequence and cache).  The sequences are
 * cut into num_chunks chunks (0: 4; at most 16 and at most B); each chunk's copies in,
 * decode and copy out run on the internal streams of csattn_attn_fwd_host, so copies
 * and kernels of different chunks overlap.
 *   seq_lens_h  read by the host during the call (each in [1, Lmax], else
 *               CSATTN_ERR_INVALID_ARG) and copied to the device asynchronously
 *   workspace   >= csattn_decode_host_workspace_size() bytes, 16-byte aligned
 * Other arguments, checks and return codes as csattn_attn_decode (max_seq_len is
 * the largest seq_lens).  Asynchronous on `stream` as csattn_attn_fwd_host; the host
 * buffers must stay valid until the work on `stream` completes.
 */
int csattn_attn_decode_host(const void* q_h, const void* k_cache_h, const void* v_cache_h,
                            const int32_t* seq_lens_h, void* out_h, int B, int Hq, int Hkv,
                            int Lmax, int d, int dtype, float scale, int num_splits,
                            int num_chunks, void* workspace, size_t workspace_bytes,
                            void* stream);

/*
 * KV-cache decode over a paged cache (the appended cache of "The Transformer
 * architecture", section "Hands-on", stored in fixed-size pages):
 *   k_pages, v_pages [num_pages, Hkv, page_size, d] bf16 (keys already rotated)
 *   block_table device int32 [B, max_pages]: row t of sequence b lives in page
 *              block_table[b * max_pages + t / page_size] at offset t % page_size
 *   q, seq_lens, out, scale, num_splits as csattn_attn_decode; max_seq_len
 *              <= max_pages * page_size
 *   workspace  >= csattn_decode_workspace_size(B, Hq, max_pages * page_size, d,
 *              num_splits) bytes
 * page_size is 16, 32 (the page is one TMA box) or a multiple of 64 up to 65536
 * (a 64-row decode tile never crosses a page).  Pages are read only for rows
 * < seq_lens[b]; a page index outside [0, num_pages)
 * raises CSATTN_ERR_DEVICE_ARG in the status word and those rows read as zeros.
 * Other errors and requirements as csattn_attn_decode.
 */
int csattn_attn_decode_paged(const void* q, const void* k_pages, const void* v_pages,
                             const int32_t* block_table, const int32_t* seq_lens, void* out, int B,
                             int Hq, int Hkv, int page_size, int num_pages, int max_pages, int d,
                             int dtype, float scale, int max_seq_len, int num_splits,
                             void* workspace, size_t workspace_bytes, void* stream);

/*
 * Bytes of device workspace csattn_attn_decode_step needs: the decode
 * partials of csattn_decode_workspace_size (rounded up to 256 bytes) followed
 * by the rotated queries, B*Hq*d*2 bytes.
 */
size_t csattn_decode_step_workspace_size(int B, int Hq, int Lmax, int d, int num_splits);

/*
 * One generation step with the cache append fused in ("The Transformer
 * architecture", section "Hands-on": the cache grows by one row per
 * generated token; the query at cache.pos sees keys 0..cache.pos; section
 * "Now: RoPE": q and k are rotated, v is not).
 *   q_new      [B, Hq, 1, d]   bf16, the new token's queries, NOT rotated
 *   k_new      [B, Hkv, 1, d]  bf16, its keys, NOT rotated
 *   v_new      [B, Hkv, 1, d]  bf16, its values
 *   k_cache, v_cache [B, Hkv, Lmax, d] bf16, caller-owned, written in place:
 *              row p_b = cache_lens[b] of every KV head receives RoPE_{p_b}(k_new)
 *              (rounded to bf16) and v_new; no other row is written
 *   cache_lens device int32 [B]: rows already cached = position of the new
 *              token; not modified (the caller advances it)
 *   out        [B, Hq, 1, d] bf16: attention of RoPE_{p_b}(q_new) over rows
 *              0..p_b, the new row included
 *   rope_base, rope_layout  as csattn_attn_fwd (rope_base <= 0: no rotation)
 *   scale, max_seq_len, num_splits  as csattn_attn_decode, where max_seq_len
 *              bounds cache_lens[b] + 1 (<= Lmax; <= 49152 with RoPE)
 *   workspace  >= csattn_decode_step_workspace_size(B, Hq, Lmax, d, num_splits)
 * Errors as csattn_attn_decode; all host-side checks run before the cache is
 * written.  A cache_lens[b] outside [0, max_seq_len - 1] raises
 * CSATTN_ERR_DEVICE_ARG in the status word and leaves that sequence's cache
 * unwritten (its output is then zero).
 */
int csattn_attn_decode_step(const void* q_new, const void* k_new, const void* v_new,
                            void* k_cache, void* v_cache, const int32_t* cache_lens, void* out,
                            int B, int Hq, int Hkv, int Lmax, int d, int dtype, float rope_base,
                            int rope_layout, float scale, int max_seq_len, int num_splits,
                            void* workspace, size_t workspace_bytes, void* stream);

/*
 * csattn_attn_decode for callers that cannot allocate device memory (for
 * example a plugin in a framework that owns all device memory and hands out
 * no allocator, or a latency-critical loop where cudaMalloc would synchronise
 * the device or could fail mid-batch).  The source pages have no counterpart
 * of this entry point; it changes only where the scratch lives.
 *
 * Same arguments and results as csattn_attn_decode, without the workspace:
 * the split partials go to a static device buffer of
 * CSATTN_DECODE_STATIC_SCRATCH_BYTES bytes that the library defines.  The
 * call allocates nothing itself (no cudaMalloc/cudaFree, no allocating
 * library call).
 *   - Argument errors (as for csattn_attn_decode) are returned before any
 *     CUDA call.  Arguments whose partials (B*Hq*splits*(d+2)*4 bytes for the
 *     split count actually used) exceed the buffer are rejected with
 *     CSATTN_ERR_WORKSPACE and a message naming both sizes; nothing is
 *     launched.  Use fewer splits, or csattn_attn_decode with a workspace.
 *   - The first call on a device is a set-up call: the CUDA runtime loads the
 *     module that holds the buffer lazily (the default module loading), so
 *     that call reserves the 16 MiB on the device and can fail with
 *     CSATTN_ERR_CUDA (out of memory); it then looks up the buffer's device
 *     address (cudaGetSymbolAddress, with that device current) and caches it.
 *     Make that first call as a warm-up before a memory pool takes the
 *     device's free memory and before any stream capture on the device;
 *     later calls reserve nothing and the device keeps the buffer until the
 *     process exits.
 *   - All calls on a device share the one buffer, which keeps the previous
 *     call's contents (nothing in it has to start at zero).  Calls whose
 *     kernels overlap on the GPU (other streams, other threads) race on it:
 *     serialise them.
 */
#define CSATTN_DECODE_STATIC_SCRATCH_BYTES (16u * 1024u * 1024u)
int csattn_attn_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                               const int32_t* seq_lens, void* out, int B, int Hq, int Hkv,
                               int Lmax, int d, int dtype, float scale, int max_seq_len,
                               int num_splits, void* stream);

/*
 * Prefill of a chunk over a paged KV cache (chunked prefill, "The Transformer
 * architecture", "Hands-on": the query at position p sees the cached keys 0..p;
 * the cache stored in fixed-size pages as for csattn_attn_decode_paged).  The
 * chunk's own keys and values are in the cache already (csattn_cache_append_paged
 * with the same cache_lens writes them).  For sequence b with L = cache_lens[b],
 * query row i sits at position L + i and, causally, sees cache rows 0..L + i
 * (all L + Tq rows with causal = 0).
 *   q          [B, Hq, Tq, d] bf16, not rotated (RoPE at positions L + i)
 *   k_pages, v_pages [num_pages, Hkv, page_size, d] bf16, keys already rotated
 *   block_table device int32 [B, max_pages]; cache_lens device int32 [B]
 *   out        [B, Hq, Tq, d] bf16;  lse NULL or fp32 [B, Hq, Tq] (natural log)
 *   rope_base, rope_layout, scale  as csattn_attn_fwd (applied to q only)
 * Requirements: bf16, d in {64, 128}, Hq % Hkv == 0, page_size 16, 32 or a multiple
 * of 64 in [64, 65536], 1 <= Tq <= max_pages * page_size < 2^24 (<= 49152 with RoPE);
 * q, pages and out 16-byte aligned, block_table, cache_lens and lse 4-byte.
 * Device-side errors (CSATTN_ERR_DEVICE_ARG in the status word): a cache_lens[b]
 * outside [0, max_pages * page_size - Tq] (that sequence's output is then not
 * meaningful; nothing is read or written out of bounds), a page index outside
 * [0, num_pages) for a row < L + Tq (those rows read as zeros).  Cache rows at or
 * past L + Tq are never used, whatever they hold.
 *   workspace  >= csattn_prefill_paged_workspace_size() bytes, 16-byte aligned
 *              (may be NULL when that is 0, i.e. for pages of 64 rows or more);
 *              16- and 32-row pages are gathered into it first, because a 128-row
 *              tile of such pages would take 4 or 8 TMA boxes in the kernel.
 * Asynchronous on `stream`.
 */
int csattn_attn_prefill_paged(const void* q, const void* k_pages, const void* v_pages,
                              const int32_t* block_table, const int32_t* cache_lens, void* out,
                              int B, int Hq, int Hkv, int Tq, int page_size, int num_pages,
                              int max_pages, int d, int dtype, int causal, float rope_base,
                              int rope_layout, float scale, float* lse, void* workspace,
                              size_t workspace_bytes, void* stream);

/*
 * Bytes of device workspace csattn_attn_prefill_paged needs: 0 for pages of 64 rows
 * or more; for 16- and 32-row pages two contiguous pools [B, Hkv, Lpad, d] bf16
 * (Lpad = max_pages * page_size rounded up to 128) and a B-entry block table, into
 * which each sequence's rows are gathered before the prefill kernel runs.
 */
size_t csattn_prefill_paged_workspace_size(int B, int Hkv, int page_size, int max_pages,
                                           int d);

/*
 * Appends Tn tokens per sequence to the KV caches (a prefill chunk written into
 * the cache, "The Transformer architecture", "Hands-on": the cache grows a row per
 * token and a token's key is rotated at its position).  For sequence b and
 * t < Tn, row r = cache_lens[b] + t receives RoPE(k_new[b, :, t]) at position r
 * (rounded to bf16 as csattn_rope_rotate rounds) and v_new[b, :, t].
 *   k_new, v_new  [B, Hkv, Tn, d] bf16 (keys not rotated)
 *   k_cache, v_cache  [B, Hkv, Lmax, d] bf16, written at rows cache_lens[b]..+Tn-1
 *   cache_lens    device int32 [B]: rows already cached (not advanced here)
 *   rope_base, rope_layout  as csattn_attn_fwd (rope_base <= 0: keys copied)
 * Requirements: bf16, d in {64, 128}, B, Hkv >= 1, 1 <= Tn <= Lmax < 2^30,
 * Tn < 2^20, Lmax <= 49152 with RoPE; pointers 16-byte aligned (cache_lens
 * 4-byte).  A sequence with cache_lens[b] < 0 or cache_lens[b] + Tn > Lmax is
 * left untouched and raises CSATTN_ERR_DEVICE_ARG in the status word.
 * Asynchronous on `stream`.
 */
int csattn_cache_append(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                        const int32_t* cache_lens, int B, int Hkv, int Tn, int Lmax, int d,
                        int dtype, float rope_base, int rope_layout, void* stream);

/*
 * csattn_cache_append into paged caches [num_pages, Hkv, page_size, d]: row r of
 * sequence b lives in page block_table[b * max_pages + r / page_size] at offset
 * r % page_size (the layout csattn_attn_decode_paged reads); the cache of a
 * sequence holds max_pages * page_size rows.  page_size is 16, 32 or a multiple of
 * 64 in [64, 65536].  A
 * page index outside [0, num_pages) raises CSATTN_ERR_DEVICE_ARG and that row is
 * not written.
 */
int csattn_cache_append_paged(const void* k_new, const void* v_new, void* k_pages, void* v_pages,
                              const int32_t* block_table, const int32_t* cache_lens, int B,
                              int Hkv, int Tn, int page_size, int num_pages, int max_pages, int d,
                              int dtype, float rope_base, int rope_layout, void* stream);

/*
 * Synchronize `stream`, then read and clear this device's status word.
 * Returns CSATTN_OK, CSATTN_ERR_TIMEOUT (a kernel wait ran out of time),
 * CSATTN_ERR_DEVICE_ARG (a device-side argument check failed) or
 * CSATTN_ERR_CUDA.
 */
int csattn_check_status(void* stream);

/*
 * Launch a one-block kernel whose wait on a barrier nothing will ever
 * complete, with a limit of `limit_us` microseconds (1..1000000).  The wait
 * runs out, the kernel returns normally and raises the timeout bit, so
 * csattn_check_status() afterwards returns CSATTN_ERR_TIMEOUT.  Exercises the
 * failure-detection path without faulting or hanging the GPU.
 */
int csattn_selftest_bounded_wait(int limit_us, void* stream);

/* Message describing the last error returned on the calling thread. */
const char* csattn_last_error(void);

/* Static name of a csattn_status value. */
const char* csattn_status_str(int status);

/* Library version, major * 10000 + minor * 100 + patch. */
int csattn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* CSATTN_H_ */
