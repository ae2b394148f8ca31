/*
 * llama_layer.h -- C ABI of libllama_layer.so: the forward pass of one
 * Llama-style decoder layer on one sm_103a GPU (prefill over a padded batch,
 * prefill over packed variable-length sequences, and KV-cache decode).
 *
 * The layer, for every token t at position p_t:
 *   x_n   = RMSNorm(x; g_in)                    RMS(a) = sqrt(mean(a^2) + eps)
 *   q,k,v = split(x_n W_qkv^T)                  rows of W_qkv: q | k | v
 *   q',k' = RoPE(q, k; p_t)                     rotate_half pairing (i, i+d/2)
 *   o     = softmax(q' k'^T / sqrt(d) + causal) v, query head h reads kv head
 *           h / (n_heads / n_kv_heads)
 *   h     = x + o W_o^T
 *   act   = silu(gate) * up, [gate | up] = RMSNorm(h; g_post) W_gate_up^T
 *   out   = h + act W_down^T
 * Sources (page title and section):
 *   - "模型层：从 Embedding 到 Loss 的实现" (nanotron tutorial ch. 9):
 *     9.3 CausalSelfAttention (fused QKV, GQA, RoPE, causal flash attention),
 *     9.4 MLP (fused gate_up, silu(gate) * up, down), 9.5 DecoderLayer
 *     (the two residual branches).
 *   - "parallel_attention.py -- LLaMA 并行注意力": 1 RoPE (inv_freq = 1 /
 *     base^(2i/d), cos/sin cache, Llama3 piecewise scaling), 2 attention
 *     (split q|k|v, repeat_kv, softmax(QK^T/sqrt(d)) V), 3 RmPad (packed
 *     tokens, cu_seqlens, causal within each sequence).
 *   - "llama3 结构详解": 3.1 RMSNorm, 3.2 Attention (the KV cache written at
 *     start_pos and read up to start_pos + seqlen).
 *   - Llama-3 model.py walkthrough (un.csdn.net): 2 RoPE (apply_scaling),
 *     3 attention with KV cache, 4 FeedForward w2(silu(w1 x) * w3 x).
 *   - NJU LLM course lecture 5: LlamaDecoderLayer shapes, RMSNorm,
 *     "RoPE高效实现" (rotate_half), SwiGLU.
 *
 * Conventions for every call:
 *   - All tensors are row-major and dense.  Element type is the config's dtype
 *     (fp32 or bf16) for x, out, weights, norm weights and the KV cache;
 *     position_ids, cu_seqlens and start_pos are int32.
 *   - Device pointers must be 16-byte aligned (x, out, weights, caches,
 *     packed, workspace) and 4-byte aligned (int32 arrays).
 *   - The library never allocates device memory: packed weights, workspace,
 *     inputs, outputs and caches belong to the caller.  It holds only a small
 *     host-side handle.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls are
 *     asynchronous on that stream.  Host-side argument checks run before any
 *     launch: a failed check returns a negative code and launches nothing.
 *   - Checks that need device data (cu_seqlens, position_ids, start_pos)
 *     run in the kernels: an offending token or sequence is skipped and a bit
 *     is set in a device status word, read by llama_layer_status().
 *   - Every wait inside a kernel is bounded; a wait that runs out sets the
 *     status word and the kernel returns (llama_layer_status reports
 *     LLAMA_ERR_DEVICE_TIMEOUT).
 *   - One layer handle serves one stream at a time: its status word, its
 *     split-tile flags, its attention work-item counters, and the copy
 *     streams and page-locked cu_seqlens buffer of llama_layer_forward_host
 *     are per handle, and a workspace holds one call's intermediates.  Calls on
 *     one stream may share a workspace (and several layers may, as the
 *     layers of a model do); concurrent calls need their own handles and
 *     workspaces.  The handle itself is not locked: call it from one host
 *     thread at a time.
 */
#ifndef LLAMA_LAYER_H
#define LLAMA_LAYER_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define LLAMA_API __attribute__((visibility("default")))
#else
#define LLAMA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes. */
#define LLAMA_OK 0
#define LLAMA_ERR_INVALID_ARG (-1)        /* null / misaligned pointer, bad size */
#define LLAMA_ERR_UNSUPPORTED_SHAPE (-2)  /* config outside the supported set */
#define LLAMA_ERR_WORKSPACE_TOO_SMALL (-3)
#define LLAMA_ERR_CUDA (-4)               /* a CUDA runtime call failed */
#define LLAMA_ERR_DEVICE_TIMEOUT (-5)     /* a bounded in-kernel wait ran out */
#define LLAMA_ERR_DEVICE_BAD_INPUT (-6)   /* bad cu_seqlens / positions / start_pos */
#define LLAMA_ERR_UNSUPPORTED_DEVICE (-7) /* not an sm_103 device */

#define LLAMA_DTYPE_F32 0
#define LLAMA_DTYPE_BF16 1

#define LLAMA_ROPE_NONE 0
#define LLAMA_ROPE_LLAMA3 1
#define LLAMA_ROPE_LINEAR 2
#define LLAMA_ROPE_DYNAMIC_NTK 3

/* Layer shape and RoPE settings.
 * Supported: head_dim in {64, 128}; n_heads % n_kv_heads == 0 and
 * n_heads / n_kv_heads <= 16;
 * hidden % 128 == 0; intermediate % 128 == 0; rms_eps > 0; rope_base > 1;
 * max_position >= 1 (length of the RoPE table: every position used must be
 * < max_position).  Llama3 scaling (see "parallel_attention.py" section 1 and
 * the model.py walkthrough section 2, apply_scaling): with wavelength
 * w_i = 2*pi / f_i, frequencies with w_i < original_max_pos / high_freq_factor
 * are kept, those with w_i > original_max_pos / low_freq_factor are divided by
 * rope_factor, and in between f_i becomes (1 - s) f_i / rope_factor + s f_i
 * with s = (original_max_pos / w_i - low) / (high - low).  Linear scaling
 * ("parallel_attention.py" section 1, t = t / scaling_factor): every f_i is
 * divided by rope_factor (> 0).  Dynamic NTK scaling (same section, the base
 * adjusted to the length; the published NTK-aware rule for a table of
 * max_position rows): when max_position > original_max_pos the base becomes
 * rope_base * (rope_factor * max_position / original_max_pos -
 * (rope_factor - 1))^(d / (d - 2)), else it is unchanged (rope_factor >= 1,
 * original_max_pos > 0).  The low / high frequency factors are read by the
 * Llama3 scaling only. */
typedef struct {
  int hidden;
  int n_heads;
  int n_kv_heads;
  int head_dim;
  int intermediate;
  float rms_eps;
  double rope_base;
  int rope_scaling; /* LLAMA_ROPE_NONE, _LLAMA3, _LINEAR or _DYNAMIC_NTK */
  double rope_factor;
  double rope_low_freq_factor;
  double rope_high_freq_factor;
  int rope_original_max_pos;
  int max_position;
  int dtype; /* LLAMA_DTYPE_F32 or LLAMA_DTYPE_BF16 */
} llama_layer_config;

/* Device pointers to the layer's weights in the pages' nn.Linear layout
 * ([out_features, in_features], row-major), element type = dtype:
 *   w_qkv     [n_heads*d + 2*n_kv_heads*d, hidden]  rows q | k | v, head-major
 *   w_o       [hidden, n_heads*d]
 *   w_gate_up [2*intermediate, hidden]              rows gate | up
 *   w_down    [hidden, intermediate]
 *   g_in, g_post [hidden]                           RMSNorm weights
 * Read only during llama_layer_init; they may be freed afterwards. */
typedef struct {
  const void *w_qkv, *w_o, *w_gate_up, *w_down, *g_in, *g_post;
} llama_layer_weights;

typedef struct llama_layer llama_layer_t;

/* Bytes of device memory llama_layer_init needs for the packed weights, the
 * RoPE table, the status word and the kernels' per-layer flags and work-item
 * counters (zeroed by llama_layer_init, left zero by every call).  Host
 * only. */
LLAMA_API int llama_layer_packed_bytes(const llama_layer_config* cfg, size_t* bytes);

/* The RoPE inverse frequencies f_i, i = 0 .. head_dim/2 - 1, the layer
 * builds its cos / sin table from (in double precision, with the scaling of
 * cfg->rope_scaling): writes head_dim / 2 values to inv_freq (host memory).
 * Validates cfg like llama_layer_packed_bytes.  Host only. */
LLAMA_API int llama_rope_inv_freq(const llama_layer_config* cfg, double* inv_freq);

/* Validates cfg, repacks the weights into `packed` (caller-owned device
 * memory of at least llama_layer_packed_bytes; it must stay allocated and
 * untouched until llama_layer_destroy), builds the RoPE cos/sin table in
 * double precision on the host and uploads it as fp32, and returns a host
 * handle in *out.  Synchronises `stream` before returning.  Repacking folds
 * g_in into the columns of W_qkv (x_n W^T = (r x) (g . W)^T with r the row's
 * 1/RMS), for bf16 layers folds g_post into the columns of W_gate_up the same
 * way (the fp32 layer keeps a copy of g_post and scales h by it), stores bf16
 * layers' weights as fp16 and interleaves the gate and up rows in blocks of
 * 128. */
LLAMA_API int llama_layer_init(const llama_layer_config* cfg,
                     const llama_layer_weights* weights, void* packed,
                     size_t packed_bytes, void* stream, llama_layer_t** out);

/* Workspace bytes for forward calls of up to `max_tokens` tokens and decode
 * calls of up to `decode_batch` sequences with caches of up to
 * `decode_max_seq` rows (pass 0 for a mode you do not use).  Host only. */
LLAMA_API int llama_layer_workspace_bytes(const llama_layer_t* layer, int max_tokens,
                                int decode_batch, int decode_max_seq,
                                size_t* bytes);

/* Prefill forward ("模型层" 9.5 DecoderLayer; "parallel_attention.py" 2 and 3).
 *   x            [total_tokens, hidden] device, input hidden states
 *   out          [total_tokens, hidden] device, output (must not alias x)
 *   position_ids [total_tokens] device int32, or NULL: positions restart at 0
 *                in every sequence.  Every position must be < max_position.
 *   cu_seqlens   NULL for a padded batch: n_seq sequences of seq_len tokens
 *                each, total_tokens == n_seq * seq_len.  Otherwise [n_seq + 1]
 *                device int32 prefix sums of the sequence lengths (packed
 *                varlen, "parallel_attention.py" 3): cu[0] = 0, non-decreasing,
 *                cu[n_seq] = total_tokens, no length above seq_len (the
 *                max_seqlen of the batch).
 * Attention is causal within each sequence.  `workspace` must hold
 * llama_layer_workspace_bytes(layer, >= total_tokens, ...). */
LLAMA_API int llama_layer_forward(llama_layer_t* layer, const void* x, void* out,
                        const int32_t* position_ids, const int32_t* cu_seqlens,
                        int n_seq, int seq_len, int total_tokens,
                        void* workspace, size_t workspace_bytes, void* stream);

/* The prefill forward with its input and output in host memory, the copies
 * overlapped with the layer: the batch is split into groups of whole
 * sequences, and while the layer runs on group i on `stream`, group i + 1 is
 * copied in and group i - 1 copied out on two streams the layer owns.
 * chunks > 0 asks for min(chunks, n_seq, LLAMA_HOST_MAX_CHUNKS) groups of
 * about equal token counts; chunks = 0 picks them: five groups of 1/16,
 * 3/16, 1/2, 3/16 and 1/16 of the tokens for a batch of at least 16384
 * tokens (small first and last groups, whose copies alone are exposed),
 * else groups of at least 2048 tokens.  Each cut falls at the first sequence
 * that starts at or after its token count, so a group may hold no rows (it
 * is skipped).  Positions restart at 0 in every sequence.
 *   x_host, out_host [total_tokens, hidden] host memory (page-locked for the
 *                    copies to be asynchronous and overlap)
 *   x_dev, out_dev   [total_tokens, hidden] device staging buffers (distinct)
 *   cu_seqlens       NULL (n_seq sequences of seq_len tokens) or HOST int32
 *                    prefix sums [n_seq + 1] under llama_layer_forward's rules
 *                    (cu[0] = 0, non-decreasing, cu[n_seq] = total_tokens, no
 *                    length above seq_len), checked on the host
 *                    (LLAMA_ERR_INVALID_ARG) and read before the call returns;
 *                    each group's copy, rebased to start at 0, is staged
 *                    through page-locked memory the layer owns into the
 *                    workspace
 * `workspace` as llama_layer_forward for total_tokens (the groups use it in
 * turn).  Returns once everything is enqueued; work enqueued on `stream`
 * afterwards runs after the last copy out, so synchronising `stream` makes
 * out_host valid.  The host buffers must stay allocated until then. */
#define LLAMA_HOST_MAX_CHUNKS 8
LLAMA_API int llama_layer_forward_host(llama_layer_t* layer, const void* x_host,
                                       void* out_host, void* x_dev, void* out_dev,
                                       const int32_t* cu_seqlens, int n_seq, int seq_len,
                                       int total_tokens, int chunks, void* workspace,
                                       size_t workspace_bytes, void* stream);

/* One decode step ("llama3 结构详解" 3.2; model.py walkthrough 3): one new
 * token per sequence.
 *   x          [batch, hidden] device, the new tokens' hidden states
 *   out        [batch, hidden] device (must not alias x)
 *   cache_k/v  [batch, max_seq, n_kv_heads, head_dim] device; rows
 *              0 .. start_pos[b]-1 hold the sequence's rotated keys / values.
 *              The new token's rotated key and its value are written at row
 *              start_pos[b]; no other row is written or read beyond it.
 *   start_pos  [batch] device int32, 0 <= start_pos[b] < max_seq and
 *              start_pos[b] < max_position; the new token's position.
 * The new token attends to cache rows 0 .. start_pos[b]. */
LLAMA_API int llama_layer_decode(llama_layer_t* layer, const void* x, void* out,
                       void* cache_k, void* cache_v, const int32_t* start_pos,
                       int batch, int max_seq, void* workspace,
                       size_t workspace_bytes, void* stream);

/* Chunked prefill with a KV cache ("llama3 结构详解" 3.2, the Meta
 * Attention.forward with start_pos and seqlen > 1; Llama-3 model.py
 * walkthrough "5. Transformer": the mask is zeros over the cached columns
 * followed by the causal triangle): seq_tokens new tokens per sequence.
 *   x          [batch * seq_tokens, hidden] device; rows b * seq_tokens ..
 *              (b + 1) * seq_tokens - 1 are sequence b's new tokens
 *   out        [batch * seq_tokens, hidden] device (must not alias x)
 *   cache_k/v  as llama_layer_decode; the new tokens' rotated keys and values
 *              are written at rows start_pos[b] .. start_pos[b] + seq_tokens - 1
 *   start_pos  [batch] device int32: the position of sequence b's first new
 *              token; every new token's position must be < max_seq and
 *              < max_position (checked on the device, status word)
 * New token i of sequence b attends to cache rows 0 .. start_pos[b] + i.
 * seq_tokens = 1 is llama_layer_decode.  Short chunks (seq_tokens <
 * LLAMA_LONG_CHUNK, e.g. checking drafted tokens) run the decode
 * projections (weights streamed once for all rows).  Their attention is the
 * split-KV attention, which reads each prefix once per group of up to
 * 16 / (n_heads / n_kv_heads) new tokens, while a sequence has at most two
 * such groups (up to 8 new tokens with 4 query heads per kv head), else the
 * tensor-core attention reading each prefix once per group of query heads.
 * Longer chunks run the prefill kernels with the tensor-core attention.  The
 * keys of cache rows past start_pos[b] + seq_tokens may be read but are
 * masked (the tensor-core attention replaces their values by zeros on chip,
 * so whatever those rows hold does not matter).
 * bf16 layers; an fp32 layer takes seq_tokens = 1 only
 * (LLAMA_ERR_UNSUPPORTED_SHAPE).  `workspace` must hold
 * llama_layer_workspace_bytes(layer, 0, >= batch * seq_tokens, >= max_seq)
 * for short chunks and llama_layer_workspace_bytes(layer, >= batch *
 * seq_tokens, 0, 0) for long ones. */
#define LLAMA_LONG_CHUNK 16
LLAMA_API int llama_layer_forward_cached(llama_layer_t* layer, const void* x, void* out,
                                         void* cache_k, void* cache_v,
                                         const int32_t* start_pos, int batch,
                                         int seq_tokens, int max_seq, void* workspace,
                                         size_t workspace_bytes, void* stream);

/* Gradient buffers of llama_layer_backward: fp32 device memory in the shapes
 * of the weights they belong to (llama_layer_weights: nn.Linear layout,
 * rows gate | up for dw_gate_up), 16-byte aligned.  Every buffer is
 * overwritten (not accumulated into). */
typedef struct {
  float *dw_qkv, *dw_o, *dw_gate_up, *dw_down;
  float *dg_in, *dg_post; /* [hidden] */
} llama_layer_grads;

/* Workspace bytes of llama_layer_backward for calls of up to `max_tokens`
 * tokens (the forward's intermediates, recomputed, plus the backward's).
 * Host only. */
LLAMA_API int llama_layer_backward_workspace_bytes(const llama_layer_t* layer,
                                                   int max_tokens, size_t* bytes);

/* Backward pass of the prefill layer: the gradients of a loss L with respect
 * to the layer's input and weights, given dL/d(out).  The pages train these
 * layers ("模型层" 9.6 LlamaForTraining puts the decoder under a loss; the
 * verl "parallel_attention.py" layers are training code) and print only the
 * forward, so every step is the chain rule applied to it, in reverse order:
 *   dW_down = dout^T act,  d act = dout W_down,
 *   d gate = d act * up * silu'(gate),  d up = d act * silu(gate),
 *   dW_gate_up = [d gate | d up]^T hn,  d hn = [d gate | d up] W_gate_up,
 *   RMSNorm^T: for y = a r g with r = (mean(a^2) + eps)^(-1/2):
 *     dg = sum over tokens of dy * a * r,  da = r (dy g) - a r^3 mean((dy g) a),
 *   dh = dout + RMSNorm^T(d hn),  dW_o = dh^T o,  d o = dh W_o,
 *   attention: P = softmax(q k^T / sqrt(d) + mask), dP = d o v^T,
 *     dz = P * (dP - rowsum(d o * o)), dq = dz k / sqrt(d),
 *     dk = dz^T q / sqrt(d), dv = P^T d o, each kv head's dk and dv summed
 *     over its n_rep query heads (the transpose of repeat_kv),
 *   RoPE^T: da = dy cos + [ (dy sin)_2, -(dy sin)_1 ] (halves of the head),
 *   dW_qkv = [dq | dk | dv]^T xn,  d xn = [dq | dk | dv] W_qkv,
 *   dx = dh + RMSNorm^T(d xn).
 * The call recomputes the forward first (nothing of the forward needs to be
 * kept by the caller) and runs on the tensor cores like the forward; bf16
 * layers only (an fp32 layer returns LLAMA_ERR_UNSUPPORTED_SHAPE).
 *   weights      the weights the layer was initialised with (device, bf16,
 *                unchanged since llama_layer_init): the norm-weight gradients
 *                read W_qkv, W_gate_up, g_in and g_post as given
 *   x            [total_tokens, hidden] device bf16, the layer's input
 *   dout         [total_tokens, hidden] device bf16, dL/d(out)
 *   dx           [total_tokens, hidden] device bf16 out, dL/dx (must alias
 *                neither x nor dout)
 *   grads        the weight gradients (fp32, see llama_layer_grads)
 *   position_ids, cu_seqlens, n_seq, seq_len, total_tokens: as
 *                llama_layer_forward
 * `workspace` must hold llama_layer_backward_workspace_bytes(layer,
 * >= total_tokens).  Gradients pass through fp16 intermediates (like the
 * forward's); scale dout so that they stay inside fp16's range, as fp16
 * training does with its loss scale. */
LLAMA_API int llama_layer_backward(llama_layer_t* layer, const llama_layer_weights* weights,
                                   const void* x, const void* dout, void* dx,
                                   const llama_layer_grads* grads,
                                   const int32_t* position_ids, const int32_t* cu_seqlens,
                                   int n_seq, int seq_len, int total_tokens, void* workspace,
                                   size_t workspace_bytes, void* stream);

/* The forward of a training step: `out` exactly as llama_layer_forward
 * computes it, and the activations the backward reads (x / RMS(x), q | k | v,
 * the attention output and its softmax denominators, h, gate | up, act and the
 * RMSNorm statistics) kept in `workspace`, so that llama_layer_backward_saved
 * can skip the forward's recomputation: a training step (forward for the
 * loss, then backward) runs the forward once instead of twice.  Arguments as
 * llama_layer_forward, except that `workspace` must hold
 * llama_layer_backward_workspace_bytes(layer, >= total_tokens).  bf16 layers
 * only (LLAMA_ERR_UNSUPPORTED_SHAPE otherwise).  The layer records the call's
 * workspace, x, position_ids, cu_seqlens, n_seq, seq_len and total_tokens
 * (host side); any later call through the layer whose workspace overlaps this
 * one drops the record. */
LLAMA_API int llama_layer_forward_train(llama_layer_t* layer, const void* x, void* out,
                                        const int32_t* position_ids,
                                        const int32_t* cu_seqlens, int n_seq, int seq_len,
                                        int total_tokens, void* workspace,
                                        size_t workspace_bytes, void* stream);

/* llama_layer_backward without the forward's recomputation: the gradients
 * from the activations the last llama_layer_forward_train call through
 * `layer` kept in `workspace`.  Arguments, results and rules as
 * llama_layer_backward; x, position_ids, cu_seqlens, n_seq, seq_len,
 * total_tokens and workspace must be the ones of that call (the pointers
 * compared as given), and the workspace not written since, else
 * LLAMA_ERR_INVALID_ARG (nothing launched).  The backward leaves the kept
 * activations intact, so it may run again from the same forward.  Enqueue it
 * on the forward's stream (or order the streams): the kept activations are
 * read on the device. */
LLAMA_API int llama_layer_backward_saved(llama_layer_t* layer,
                                         const llama_layer_weights* weights, const void* x,
                                         const void* dout, void* dx,
                                         const llama_layer_grads* grads,
                                         const int32_t* position_ids,
                                         const int32_t* cu_seqlens, int n_seq, int seq_len,
                                         int total_tokens, void* workspace,
                                         size_t workspace_bytes, void* stream);

/* Self-test of the bounded waits the library's pipelined kernels use (no
 * layer needed): one block waits on an mbarrier that nothing arrives on and
 * on a device flag that nothing sets, each up to the library's wait limit
 * (2 s).  Synchronises `stream` and writes observed[0] / observed[1] = 1 if
 * the mbarrier / flag wait completed, 0 if it gave up, and observed[2] = the
 * status word the waits wrote (bit 1: a wait ran out).  A working build gives
 * {0, 0, 1} and leaves the context usable.  Returns LLAMA_OK, or
 * LLAMA_ERR_CUDA if the launch or the copy fails. */
LLAMA_API int llama_selftest_bounded_waits(int observed[3], void* stream);

/* Synchronises `stream`, reads and clears the device status word.  Returns
 * LLAMA_OK, LLAMA_ERR_DEVICE_TIMEOUT or LLAMA_ERR_DEVICE_BAD_INPUT. */
LLAMA_API int llama_layer_status(llama_layer_t* layer, void* stream);

/* Byte offsets inside the workspace of the intermediates of the last call
 * with these sizes, for checking individual stages:
 *   [0] q|k|v after RoPE   [tokens, n_heads*d + 2*n_kv_heads*d]
 *   [1] attention output    [tokens, n_heads*d]
 *   [2] h (after o_proj + residual) [tokens, hidden]
 *   [3] act = silu(gate)*up [tokens, intermediate]
 * Element types: fp32 layers keep everything in fp32.  bf16 layers (bf16
 * input, weights, output and cache) keep their intermediates in fp16, which
 * holds bf16 values exactly and rounds 8x finer: q|k|v is fp16 for
 * llama_layer_forward and bf16 for llama_layer_decode (it is written to the
 * bf16 cache); the attention output is fp16; h is fp16 holding h / 256 (the
 * MLP input and the residual of down_proj); act is fp16 holding act / 16.
 * decode == 1 gives the decode layout (tokens <= 256). */
#define LLAMA_WS_NUM 4
LLAMA_API int llama_layer_workspace_offsets(const llama_layer_t* layer, int tokens,
                                  int decode, size_t offsets[LLAMA_WS_NUM]);

/* Stage timing.  With timing on, every forward / decode call records a CUDA
 * event on its stream where each of its stages begins and one where the call
 * ends, into the next record of a ring of `ring_calls` records (events are
 * driver objects, not device memory).  ring_calls = 0 switches timing off
 * (the default); 1 <= ring_calls <= LLAMA_MAX_TIMED_CALLS switches it on and
 * forgets earlier records.  Returns LLAMA_ERR_CUDA if the events cannot be
 * created. */
#define LLAMA_MAX_STAGES 16
#define LLAMA_MAX_TIMED_CALLS 4096
LLAMA_API int llama_layer_set_timing(llama_layer_t* layer, int ring_calls);

/* Stage durations of a recorded call, in milliseconds
 * (cudaEventElapsedTime between consecutive events; waits for that call's
 * last event).  call = 0 is the most recent forward / decode call, 1 the one
 * before, ... (< ring_calls).  Writes up to max_stages entries of ms[] and of
 * names[] (static strings; names may be NULL) and the number of stages in
 * *n_stages (may be NULL): 0 when timing is off or the call was not recorded,
 * at most LLAMA_MAX_STAGES (the first ones of a call that has more).  Stages
 * of a prefill: "rmsnorm_stats", "qkv_rope", "attention", "o_proj_residual",
 * "gate_up_swiglu", "down_residual"; a backward call adds its own stages
 * (names starting with "bwd_"). */
LLAMA_API int llama_layer_stage_times(llama_layer_t* layer, int call,
                                      int max_stages, float* ms,
                                      const char** names, int* n_stages);

/* Number of kernels the last forward / decode call launched (timing on or
 * off), or LLAMA_ERR_INVALID_ARG for a null handle. */
LLAMA_API int llama_layer_launch_count(const llama_layer_t* layer);

/* Frees the host handle only (packed memory stays the caller's). */
LLAMA_API void llama_layer_destroy(llama_layer_t* layer);

/* Static string for a return code. */
LLAMA_API const char* llama_layer_strerror(int code);

/* out = bf16(x / RMS(x) * g) per row, RMS(x) = sqrt(mean(x^2) + eps): the
 * model's final RMSNorm before the output projection ("模型层" 9.5; Llama-3
 * model.py walkthrough "5. Transformer", self.norm then self.output).  x, out
 * [rows, hidden] bf16 and g [hidden] bf16, device, 16-byte aligned, out must
 * not alias x; hidden % 128 == 0; fp32 arithmetic, one rounding. */
LLAMA_API int llama_rmsnorm_bf16(const void* x, const void* g, void* out, int rows,
                                 int hidden, float eps, void* stream);

/* D[M, N] = A[M, K] . B[N, K]^T in bf16 with fp32 accumulation, on the same
 * tcgen05 / TMA GEMM the layer's projections use (the contraction of every
 * nn.Linear on the pages, and the model's output projection to the vocabulary
 * logits).  A, B, D device, row-major, 16-byte aligned; K % 8 == 0,
 * N % 32 == 0.  The kernel's bounded waits report into a status word of the
 * current device that llama_gemm_status reads. */
LLAMA_API int llama_gemm_bf16(const void* A, const void* B, void* D, int M, int N, int K,
                    void* stream);

/* Synchronises `stream`, then reads and clears the status word of the
 * standalone GEMMs (llama_gemm_bf16, llama_gemm_bf16_streamk_static) on the
 * current device: a bounded wait inside one of them that ran out (its output
 * is then incomplete) gives LLAMA_ERR_DEVICE_TIMEOUT.  The word is shared by
 * every standalone GEMM on the device since the last read.  Returns LLAMA_OK,
 * LLAMA_ERR_DEVICE_TIMEOUT or LLAMA_ERR_CUDA. */
LLAMA_API int llama_gemm_status(void* stream);

/* D[M, N] = A[M, K] . B[N, K]^T in bf16 with fp32 accumulation, without any
 * device memory from the caller beyond A, B and D.  The pages this library
 * follows have no counterpart of this entry point: it exists for callers that
 * cannot allocate device memory where they run the GEMM (an engine that has
 * reserved all device memory for its own pool, or a latency-critical loop in
 * which cudaMalloc / cudaFree could synchronise the device) and have no
 * workspace to hand over.
 *
 * It runs the stream-K tcgen05 GEMM of the decode projections (A is the
 * large side, e.g. a weight matrix; B holds up to 256 rows, e.g. tokens; K
 * is split evenly over all SMs) and keeps the fp32 partial sums in a 16 MiB
 * array of device memory that the library defines at file scope: every GPU
 * that loads the library holds those 16 MiB until the process exits.  The
 * partials of tile t fill slots x 128 x bn floats (bn = 64, 128 or 256, the
 * smallest >= N); a call whose partials need more than 16 MiB returns
 * LLAMA_ERR_WORKSPACE_TOO_SMALL and launches nothing.
 *   A [M, K], B [N, K], D [M, N]: device, row-major, 16-byte aligned;
 *   K % 8 == 0, N % 8 == 0, N <= 256 (else LLAMA_ERR_UNSUPPORTED_SHAPE).
 * The first call on a device (with that device current) looks up the
 * array's device address with cudaGetSymbolAddress; make that first call
 * before any stream capture.  The call never calls cudaMalloc, cudaFree or
 * an allocating library routine.  Every call shares the one array, which
 * keeps the last call's partials; a call writes every partial it reads, so
 * nothing has to start at zero.  Calls that overlap on the GPU (other
 * streams, other host threads) race on the array: order them on one stream.
 * A bounded wait of the GEMM that runs out is not returned by this call (it
 * returns once the kernels are enqueued): llama_gemm_status reports it. */
LLAMA_API int llama_gemm_bf16_streamk_static(const void* A, const void* B, void* D,
                                             int M, int N, int K, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* LLAMA_LAYER_H */
