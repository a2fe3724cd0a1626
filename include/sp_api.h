/*
 * sp_api.h — C ABI of the sequence-parallel (Ulysses-style) attention step
 * for one GB300 (sm_103a), with W "virtual ranks" held in W disjoint device
 * buffers on the same GPU.
 *
 * The step follows "LTX-2 序列并行拆解: token 切分、all2all 换头与 runner 接入全链路"
 * (LTX-2 sequence-parallel breakdown):
 *   补齐 (pad)          sp_pad, sp_pad_mask
 *   切分 (partition)    sp_partition, sp_tile
 *   换头 (head swap)    sp_send_recv_heads, sp_attention, sp_gather_heads;
 *                       sp_attention_shards (the exchange fused into the
 *                       attention); sp_pad_send_heads / sp_gather_heads_output
 *                       (the exchange fused with its neighbours)
 *   还原 (restore)      sp_gather_output, sp_unpad
 * and the kernel paragraphs on SM rotation ("SM 轮转") and the completion
 * barrier ("barrier").  An alternative partition for the tile step follows
 * the LongCat-Video context-parallel page (智能张量拆分, 2-D tensor split):
 * sp_optimal_split, sp_tile_2d, sp_gather_2d.
 *
 * Conventions shared by every entry point
 *   - Activations are row-major [B, T, H, D] ("tokens x heads x head_dim").
 *     Rank r owns the token block [r*Tl, (r+1)*Tl) and the head block
 *     [r*Hl, (r+1)*Hl) with Tl = T_pad / W and Hl = H / W.
 *   - Masks are uint8, 1 = the query may attend to the key.
 *   - Every tensor pointer is a DEVICE pointer owned by the caller; arrays of
 *     W per-rank pointers ("void* const* shards") are HOST arrays holding
 *     device pointers.  The library allocates no device memory: the caller
 *     passes a zero-initialised workspace where one is needed.
 *   - Every call is asynchronous on the caller's stream (a cudaStream_t,
 *     passed as sp_stream_t; NULL = the legacy default stream) and is ordered
 *     only by that stream.
 *   - Every call validates its arguments on the host and returns an sp_status
 *     code; nothing is thrown across the ABI.  sp_last_error() gives a
 *     thread-local message for the last failing call on this thread.
 *     Errors raised on the device (a failed completion-barrier check, a
 *     bounded wait that ran out) are recorded in the workspace's status word
 *     and read with sp_workspace_status().
 *   - Buffers of one call must not overlap unless stated.
 */
#ifndef SP_API_H
#define SP_API_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *sp_stream_t; /* == cudaStream_t */

/* Symbols of this header are the library's only exports. */
#if defined(__GNUC__)
#define SP_API __attribute__((visibility("default")))
#else
#define SP_API
#endif

/* Peer cap of the pages' IPC all-to-all kernel (MAX_NUM_PEERS = 8, section
 * "直写"); the virtual ranks keep the same cap. */
#define SP_MAX_RANKS 8

typedef enum {
    SP_OK = 0,
    SP_ERR_NOT_DIVISIBLE = 1,       /* total tokens not a multiple of W (切分: ValueError) */
    SP_ERR_HEADS_NOT_DIVISIBLE = 2, /* H not a multiple of W (换头 gives each rank H/W heads) */
    SP_ERR_INVALID_ARG = 3,         /* null pointer, negative size, W out of [1, SP_MAX_RANKS] */
    SP_ERR_ALIGNMENT = 4,           /* pointer or stride alignment a kernel needs is not met */
    SP_ERR_UNSUPPORTED = 5,         /* dtype / head_dim combination not built */
    SP_ERR_TIMEOUT = 6,             /* a bounded device wait ran out (device status) */
    SP_ERR_BARRIER = 7,             /* completion counters disagree with the CTA map (device status) */
    SP_ERR_CUDA = 8                 /* a CUDA runtime call failed; see sp_last_error() */
} sp_status;

typedef enum { SP_F32 = 0, SP_BF16 = 1 } sp_dtype;

typedef enum {
    SP_MASK_NONE = 0, /* every key visible */
    SP_MASK_KEY = 1,  /* key-only mask, uint8 [Tk]: the (1,1,T_padded) mask of 补齐 */
    SP_MASK_FULL = 2  /* full mask, uint8 [B, Tq, Tk] (row-major, contiguous) */
} sp_mask_kind;

/* Size in bytes of the workspace header every exchange call needs.  The
 * caller zero-fills it once; calls leave it ready for the next call. */
#define SP_WORKSPACE_HEADER_BYTES 256

/* Fault injection for tests of the device-side timeouts (no counterpart in
 * the pages): the int32 at this byte offset of a workspace is 0 in normal
 * use.  A positive value k makes the tensor-core attention kernel that uses
 * the workspace issue only its first k - 1 K/V tile loads, so its bounded
 * waits run out (2 s each): the call then leaves SP_ERR_TIMEOUT in the
 * status word, every CTA drains what it had in flight and exits, and the
 * context stays usable.  Nothing faults and nothing waits without a bound. */
#define SP_WORKSPACE_KV_STALL_OFFSET 80

/* Human-readable name of a status code (static string). */
SP_API const char *sp_status_string(int status);
/* Thread-local message describing the last failing call on this thread. */
SP_API const char *sp_last_error(void);
/* ABI version; bumps on incompatible changes. */
SP_API int sp_version(void);
/* Number of CUDA kernels this library has launched in this process (all
 * threads, all devices); a host-side counter for accounting and tests. */
SP_API uint64_t sp_launch_count(void);

/* ----------------------------------------------------------------------
 * 补齐 (pad).  T_pad = the smallest multiple of W that is >= T.
 * Host only.  Returns SP_ERR_INVALID_ARG for T < 0, W < 1 or T_pad == NULL. */
SP_API int sp_padded_len(int T, int W, int *T_pad);

/* x [B, T, row_bytes] -> x_pad [B, T_pad, row_bytes]: rows t >= T are zero.
 * row_bytes = H*D*element size.  T_pad >= T.  x and x_pad must not overlap. */
SP_API int sp_pad(const void *x, void *x_pad, int B, int T, int T_pad, int64_t row_bytes,
           sp_stream_t stream);

/* Padding mask.
 *   user_mask == NULL: mask_out is the key-only mask (1,1,T_pad):
 *       mask_out[k] = (k < T).  O(T) memory, the (B,T,T) matrix is never built.
 *   user_mask != NULL: user_mask is (B, T, T); mask_out is (B, T_pad, T_pad):
 *       mask_out[b,q,k] = user_mask[b,q,k]  for q < T and k < T,
 *                       = 1                 for q >= T and k < T (a pad query
 *                         row keeps visibility of the valid keys, so no pad row
 *                         is fully masked and none yields NaN),
 *                       = 0                 for k >= T. */
SP_API int sp_pad_mask(const uint8_t *user_mask, uint8_t *mask_out, int B, int T, int T_pad,
                sp_stream_t stream);

/* ----------------------------------------------------------------------
 * 切分 (partition).  Uniform shards: total_tokens must divide by W, else
 * SP_ERR_NOT_DIVISIBLE (the page's ValueError).  Host only.
 * starts[r] = r*Tl and lens[r] = Tl for r < W (arrays of W ints, host). */
SP_API int sp_partition(int total_tokens, int W, int *starts, int *lens);

/* tile_modality_for_rank for activations: x_pad [B, T_pad, row_bytes] ->
 * shards[r] [B, Tl, row_bytes] holding tokens [r*Tl, (r+1)*Tl).
 * SP_ERR_NOT_DIVISIBLE if T_pad % W != 0. */
SP_API int sp_tile(const void *x_pad, void *const *shards, int W, int B, int T_pad, int64_t row_bytes,
            sp_stream_t stream);

/* ----------------------------------------------------------------------
 * 2-D spatial split: an alternative partition for the tile step, after the
 * LongCat-Video context-parallel page, section 智能张量拆分 (2-D tensor split).
 * The latent tokens of a batch item form a row-major [F, Hg, Wg] grid
 * (frames x patch rows x patch columns; T = F*Hg*Wg).  The world size is
 * factored as split_h x split_w, the factor pair closest to a square with the
 * smaller factor on height (sp_optimal_split).  Every frame is cut into
 * split_h bands of Hg/split_h rows and every band into split_w pieces of
 * Wg/split_w columns; rank r = ih*split_w + iw holds piece (ih, iw) of every
 * frame, tokens in (frame, row, column) order:
 *
 *   shards[ih*split_w + iw][b, (f*bh + h)*bw + w, :] = x[b, (f*Hg + ih*bh + h)*Wg + iw*bw + w, :]
 *
 * Every rank then holds Tl = F*bh*bw tokens, so sp_send_recv_heads,
 * sp_attention and sp_gather_heads run unchanged on these shards (the
 * attention sees the keys in another order, which changes only the order of
 * the key sum).
 */

/* (split_h, split_w) with split_h * split_w = W, split_w - split_h minimal,
 * split_h <= split_w.  Host only.  SP_ERR_INVALID_ARG for W < 1. */
SP_API int sp_optimal_split(int W, int *split_h, int *split_w);

/* x [B, F*Hg*Wg, row_bytes] -> shards[r] [B, F*(Hg/split_h)*(Wg/split_w),
 * row_bytes], r < split_h*split_w <= SP_MAX_RANKS.  SP_ERR_NOT_DIVISIBLE if
 * Hg % split_h or Wg % split_w is not 0 (the blocks must be uniform, as the
 * token-range partition requires). */
SP_API int sp_tile_2d(const void *x, void *const *shards, int B, int F, int Hg, int Wg, int split_h, int split_w,
                      int64_t row_bytes, sp_stream_t stream);

/* The inverse of sp_tile_2d: every rank's piece back to its place in
 * out [B, F*Hg*Wg, row_bytes].  Same argument rules. */
SP_API int sp_gather_2d(const void *const *shards, void *out, int B, int F, int Hg, int Wg, int split_h,
                        int split_w, int64_t row_bytes, sp_stream_t stream);

/* ----------------------------------------------------------------------
 * 换头 (head exchange), the token x head all-to-all, run as an on-device
 * permutation between the W virtual-rank buffers.
 *
 *   heads[r][b, s*Tl + t, h', :] = shards[s][b, t, r*Hl + h', :]
 *
 * shards[s]: [B, Tl, H, D], heads[r]: [B, W*Tl, Hl, D]; elt_bytes is the
 * element size (1, 2, 4 or 8).  Every (source rank, token, destination rank)
 * piece is a contiguous run of Hl*D*elt_bytes bytes.
 *
 * SM rotation (section "SM 轮转"): CTA i of the launch writes destination
 * rank i % W and its rank group walks all of that rank's tokens with a
 * stride, so ranks get CTA counts that differ by at most one when the CTA
 * count is not a multiple of W.
 * Barrier (section "barrier"): after its writes, every CTA atomically
 * increments its destination rank's counter in the workspace; the last CTA
 * to finish checks every counter against the CTA map, records the counts,
 * resets the counters and sets SP_ERR_BARRIER in the status word on a
 * mismatch.  Nothing on the device waits: on one GPU, stream order already
 * orders the consumer kernel after this one.
 *
 * workspace: device, >= SP_WORKSPACE_HEADER_BYTES, 16-byte aligned,
 * zero-filled before its first use; calls that share a workspace must not
 * overlap on the device.
 * Errors: SP_ERR_HEADS_NOT_DIVISIBLE if H % W != 0; SP_ERR_INVALID_ARG. */
SP_API int sp_send_recv_heads(const void *const *shards, void *const *heads, int W, int B, int Tl, int H,
                       int D, int elt_bytes, void *workspace, sp_stream_t stream);

/* gather_heads, the exact inverse of sp_send_recv_heads:
 *   shards[s][b, t, r*Hl + h', :] = heads[r][b, s*Tl + t, h', :]
 * Same SM rotation (CTA i reads source rank i % W) and barrier. */
SP_API int sp_gather_heads(const void *const *heads, void *const *shards, int W, int B, int Tl, int H,
                    int D, int elt_bytes, void *workspace, sp_stream_t stream);

/* The exchange fused with its neighbours on one GPU, where the token shards
 * need not exist: pad and tile fused with the send, the inverse exchange
 * fused with gather_output.  Same bytes as the staged calls (sections 补齐,
 * 切分, 换头, 还原), one pass over the data instead of three.
 *
 * sp_pad_send_heads = sp_pad + sp_tile + sp_send_recv_heads in one pass over
 * the caller's x [B, T, H, D]:
 *   heads[r][b, g, h', :] = x[b, g, r*Hl + h', :]  for g < T,  0 for T <= g < T_pad.
 * heads[r]: [B, T_pad, Hl, D].  T <= T_pad; T_pad % W != 0 gives
 * SP_ERR_NOT_DIVISIBLE, H % W != 0 SP_ERR_HEADS_NOT_DIVISIBLE.  Same SM
 * rotation, completion counters and workspace rules as sp_send_recv_heads. */
SP_API int sp_pad_send_heads(const void *x, void *const *heads, int W, int B, int T, int T_pad, int H, int D,
                             int elt_bytes, void *workspace, sp_stream_t stream);

/* sp_gather_heads_output = sp_gather_heads + sp_gather_output (cropped to
 * T_out, which is the unpad when T_out = T) in one pass:
 *   out[b, g, r*Hl + h', :] = heads[r][b, g, h', :]  for g < T_out <= T_pad.
 * out: [B, T_out, H, D].  Same rotation, counters and workspace rules. */
SP_API int sp_gather_heads_output(const void *const *heads, void *out, int W, int B, int T_pad, int T_out, int H,
                                  int D, int elt_bytes, void *workspace, sp_stream_t stream);

/* sp_send_recv_heads without a caller workspace, for callers that cannot
 * allocate device memory: for example a plugin that is handed tensors by a
 * host framework whose allocator it cannot reach, or an inference loop that
 * must run inside a fixed, preallocated memory budget.  The paper has no
 * counterpart: this is a convenience of this library.
 *
 * Same arguments, layout and result as sp_send_recv_heads.  The exchange's
 * scratch (status word, finish ticket and the per-destination completion
 * counters, SP_WORKSPACE_HEADER_BYTES = 256 bytes) lives in one static device
 * array inside the library; every GPU that loads the library holds those 256
 * bytes until the process exits.  The array covers at most SP_MAX_RANKS
 * destination ranks: W > SP_MAX_RANKS is rejected with SP_ERR_INVALID_ARG.
 * Nothing is allocated: no cudaMalloc, no cudaFree, no allocating library call.
 *
 * The first call on a device looks up the array's device address on that
 * device (cudaGetSymbolAddress), so make the first call on each device before
 * any stream capture begins.  Every argument is checked first: a rejected call
 * returns its error and leaves the array untouched.  A call that passes the
 * checks clears the finish ticket and the counters on `stream` before its
 * kernel runs; the status word is kept.  All calls share the one array: calls
 * that overlap on the GPU (other streams, other host threads) race on it;
 * serialise them.
 * status_out (host, may be NULL): when given, the call waits for `stream`,
 * stores the status word there -- the first device error (SP_ERR_BARRIER)
 * recorded by any exchange on this device since the last read, else SP_OK --
 * and resets it to SP_OK; when NULL the call stays asynchronous and an error
 * it records waits for the next call that reads the status. */
SP_API int sp_send_recv_heads_noalloc(const void *const *shards, void *const *heads, int W, int B, int Tl,
                                      int H, int D, int elt_bytes, int *status_out, sp_stream_t stream);

/* Reads the workspace header (synchronises `stream`).  *status gets the
 * sticky device status (SP_OK or the first device error since the last
 * clear); counts (may be NULL) gets the per-destination CTA counts the last
 * completed exchange observed (SP_MAX_RANKS ints); n_launches (may be NULL)
 * gets the number of completed exchange launches.  clear != 0 resets the
 * status word to SP_OK. */
SP_API int sp_workspace_status(void *workspace, int *status, int *counts, int *n_launches, int clear,
                        sp_stream_t stream);

/* Host helper: CTA counts per destination rank that the exchange's SM
 * rotation gives for a grid of n_ctas CTAs (counts: W ints). */
SP_API int sp_sm_rotation_counts(int n_ctas, int W, int *counts);

/* Number of CTAs the exchange kernels launch on the current device. */
SP_API int sp_exchange_grid(int *n_ctas);

/* ----------------------------------------------------------------------
 * Attention on the local heads (section 换头).  For each rank r, batch b,
 * local head h and query q:
 *   s_k   = scale * sum_d Q_r[b,q,h,d] * K_r[b,k,h,d]     over visible keys k
 *   O_r[b,q,h,:] = sum_k softmax(s)_k * V_r[b,k,h,:]
 * Keys k >= Tk are never visible; a row with no visible key yields 0.
 * One launch covers all W ranks x B x Hl heads x query tiles.
 *
 * q/k/v/o: host arrays of W device pointers to element [b=0, t=0, h=0, d=0]
 * of each rank's tensor.  Strides (host arrays of 3 int64, in ELEMENTS:
 * batch, token, head; d is contiguous) describe each tensor; NULL means the
 * contiguous [B, T, Hl, D] layout.  Example: the cross-attention query kept
 * whole on every rank ([B, Tq, H, D], sliced to the rank's heads in place)
 * passes q[r] = Q + r*Hl*D and q_strides = {Tq*H*D, H*D, D}.
 *
 * dtype: SP_F32 (fp32 in, fp32 accumulate, fp32 out) or SP_BF16 (bf16 in,
 * fp32 accumulate, bf16 out rounded to nearest even).  bf16 with D = 64 or
 * 128 and 16-byte aligned strides runs on the tcgen05 tensor-core kernel;
 * other shapes run on a CUDA-core kernel (D <= 256).
 * mask: see sp_mask_kind (device pointer, NULL for SP_MASK_NONE).
 * scale <= 0 selects 1/sqrt(D).
 * workspace: device, zero-filled before first use, >= the size returned by
 * sp_attention_workspace_bytes() for the same shape (it holds the status word
 * and the partial results of a split-key pass for short query sequences).
 * A workspace smaller than that but >= SP_WORKSPACE_HEADER_BYTES runs the
 * kernel without the split.  Calls sharing a workspace must not overlap. */
SP_API int sp_attention(const void *const *q, const void *const *k, const void *const *v, void *const *o,
                 int W, int B, int Tq, int Tk, int Hl, int D, sp_dtype dtype,
                 const int64_t *q_strides, const int64_t *kv_strides, const int64_t *o_strides,
                 sp_mask_kind mask_kind, const uint8_t *mask, float scale, void *workspace,
                 size_t workspace_bytes, sp_stream_t stream);

/* The head exchange fused into the attention (one GPU): sp_send_recv_heads
 * only moves each rank's heads of every source shard into one buffer; here
 * the attention's tile loads read them where they are (sections 换头 and
 * 直写: the data goes straight to its consumer, with no intermediate copy).
 *
 * A sharded operand of T tokens (Tq for q/o, Tk for k/v) is given as its W
 * source-rank token shards, Tl = ceil(T / W) tokens apart: shard s holds
 * tokens [s*Tl, s*Tl + n_s) in its first n_s = clamp(T - s*Tl, 0, Tl) rows,
 * all H heads ([B, >= n_s, H, D], strides as below).  These may be views of
 * the caller's unpadded [B, T, H, D] tensor -- the last shards then stop at
 * token T, and a shard with n_s = 0 may be NULL -- or padded [B, Tl, H, D]
 * buffers passed with T = W*Tl.  Rows past n_s are never read or written, so
 * no padding and no padding mask is needed; masks index real tokens
 * (SP_MASK_KEY: [Tk], SP_MASK_FULL: [B, Tq, Tk]).
 *
 * Rank r's local head h is head r*Hl + h of every shard.  Its keys are
 * visited as every shard's whole 128-row tiles (loaded by TMA from the
 * shard), then each shard's leftover block of n_s % 128 rows: by TMA as a
 * partial tile when it holds at least 64 rows (the rows past the shard's end
 * read as zeros and are masked), else packed with the other small leftover
 * blocks into "gathered" tiles copied row by row; queries are tiled the same
 * way and O rows go back to their shard.  Attention does not depend on the order of
 * its keys, so only the rounding of the key sum differs from sp_attention on
 * the exchanged (padded, key-masked) tensors; when Tl is a multiple of 128
 * the tiles are exactly the exchanged layout's and the result is the same
 * bit for bit.
 *
 * shard_flags: SP_SHARD_KV -- k[s], v[s] are shards (strides kv_strides, or
 * NULL for contiguous [B, Tl, H, D]); SP_SHARD_Q -- q[s], o[s] are shards read
 * and written in place (o[s] then receives every rank's heads of shard s, the
 * layout sp_gather_heads produces).  An operand without its flag is per rank
 * as in sp_attention: [B, T, H/W, D] views with their strides.
 * H is the total head count (H % W == 0, else SP_ERR_HEADS_NOT_DIVISIBLE);
 * bf16 with D = 64 or 128 only (else SP_ERR_UNSUPPORTED), 16-byte aligned
 * pointers and strides (else SP_ERR_ALIGNMENT); Tk = 0 gives
 * SP_ERR_UNSUPPORTED.  Scale, workspace (sp_attention_workspace_bytes with
 * Hl = H/W and these Tq, Tk) and status as sp_attention.  When the shards'
 * leftover blocks add tiles (up to W more than ceil(T / 128)), a last wave
 * that would want more split partials than that workspace holds runs whole. */
#define SP_SHARD_KV 1
#define SP_SHARD_Q 2
SP_API int sp_attention_shards(const void *const *q, const void *const *k, const void *const *v, void *const *o,
                               int W, int B, int Tq, int Tk, int H, int D, sp_dtype dtype, int shard_flags,
                               const int64_t *q_strides, const int64_t *kv_strides, const int64_t *o_strides,
                               sp_mask_kind mask_kind, const uint8_t *mask, float scale, void *workspace,
                               size_t workspace_bytes, sp_stream_t stream);

/* Workspace bytes sp_attention wants for this shape on the current device. */
SP_API size_t sp_attention_workspace_bytes(int W, int B, int Tq, int Tk, int Hl, int D, sp_dtype dtype);

/* ----------------------------------------------------------------------
 * 还原 (restore).  gather_output_tokens: each rank's local output is padded
 * to the longest shard (a no-op: shards are uniform), all shards are
 * gathered, each rank's piece is cropped to its real token count
 *   n_r = clamp(T_out - r*Tl, 0, Tl)
 * and the pieces are concatenated:
 *   out[b, r*Tl + t, :] = shards[r][b, t, :]   for r*Tl + t < T_out.
 * shards[r]: [B, Tl, row_bytes]; out: [B, T_out, row_bytes], T_out <= W*Tl.
 * T_out = W*Tl gives the padded sequence; T_out = T (the caller's length)
 * crops and unpads in the same pass. */
SP_API int sp_gather_output(const void *const *shards, void *out, int W, int B, int Tl, int T_out,
                     int64_t row_bytes, sp_stream_t stream);

/* unpad: x_pad [B, T_pad, row_bytes] -> out [B, T, row_bytes], T <= T_pad. */
SP_API int sp_unpad(const void *x_pad, void *out, int B, int T_pad, int T, int64_t row_bytes,
             sp_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SP_API_H */
