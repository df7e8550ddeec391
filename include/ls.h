/* ls.h — C ABI of the layer-streamed NF4 LoRA fine-tuning library (libls.so).
 *
 * What it computes: one training step of plain-LoRA fine-tuning over a frozen,
 * NF4-quantised decoder base that lives in pinned host RAM and is copied to the GPU
 * one decoder layer at a time on a dedicated copy stream ("The Core Idea: Layer
 * Streaming" and the FAQ of Soup: Fine-Tune an 8B Model on a 4 GB GPU).  Two device
 * slots are double-buffered: layer l+1 is copied while layer l computes, so peak
 * device memory is two layer slots, the activation store and the adapter.  SFT uses
 * next-token cross-entropy; DPO takes its reference logprobs from a second pass over
 * the same streamed base with the adapter switched off (Show HN: Fine-tune an 8B
 * model on a 4 GB laptop GPU, first paragraph; the evermx.com summary), so there is
 * no second copy of the weights.  A forward pass may also run "resident" (every
 * layer kept on the device); streamed and resident results are bit-identical, the
 * pages' correctness bar (axbrief.com, "Beyond Memory: The Layer Streaming
 * Breakthrough").
 *
 * Conventions
 *  - Every function returns an int status: LS_OK (0) or a negative LS_ERR_*.
 *    Errors on a context are sticky: once a call fails, later calls on the same
 *    context return the same code; ls_last_error() gives the message.
 *  - Pointers named d_* are device pointers; h_* are host pointers.  The caller owns
 *    every buffer it passes in and keeps it alive for as long as the text says.
 *  - Device work is enqueued asynchronously on the caller's compute stream; host
 *    pinned-memory copies on the caller's copy stream.  ls_plan, nf4_quantize,
 *    ls_stats and ls_last_error are synchronous host calls; ls_sync waits.
 *  - The library never allocates device memory: ls_plan reports the workspace size,
 *    the caller allocates it (e.g. through PyTorch) and hands it to ls_create.
 *  - bf16 values travel as uint16_t bit patterns; matrices are dense row-major.
 *  - There is no CPU fallback: without a CUDA device every compute call fails.
 */
#ifndef LS_H_
#define LS_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  LS_OK = 0,
  LS_ERR_ARG = -1,      /* an argument is outside the documented contract            */
  LS_ERR_CAP = -2,      /* pre-flight: the run does not fit the device memory cap     */
  LS_ERR_CUDA = -3,     /* a CUDA runtime call failed                                 */
  LS_ERR_TIMEOUT = -4,  /* a host-side bounded wait (ls_sync) ran out                 */
  LS_ERR_STATE = -5,    /* call out of order (e.g. backward without a saved forward) */
  LS_ERR_DEVICE = -6    /* a kernel raised the device error flag (bounded wait lost)  */
};

/* Shape and run parameters of a Llama-style stack (pre-norm RMSNorm, bias-free
 * q/k/v/o, rotate-half RoPE, causal grouped-query attention, SwiGLU MLP). */
typedef struct ls_config {
  int32_t layers;          /* decoder layers L                                        */
  int32_t hidden;          /* H, multiple of 64                                       */
  int32_t heads;           /* query heads nh                                          */
  int32_t kv_heads;        /* key/value heads (nh % kv_heads == 0)                    */
  int32_t head_dim;        /* 64 or 128                                               */
  int32_t inter;           /* SwiGLU inner size I, multiple of 64                     */
  int32_t vocab;           /* V, multiple of 64                                       */
  int32_t tied;            /* 1: the embedding matrix is also the vocabulary head     */
  int32_t lora_r;          /* LoRA rank, 1..16 (q_proj and v_proj)                    */
  float lora_scale;        /* s = alpha / r                                           */
  float rope_theta;
  float eps;               /* RMSNorm epsilon                                         */
  int32_t max_tokens;      /* upper bound on tokens per pass (T)                      */
  int32_t max_seqs;        /* upper bound on sequences per pass                       */
  int32_t max_seq_len;     /* longest sequence (RoPE table rows); 0 = max_tokens      */
  int32_t vocab_chunk_rows;/* rows of the vocabulary head per streamed chunk; 0 = auto */
  int32_t resident;        /* 1: keep every layer on the device (test/reference mode) */
  int32_t dpo_shared_read; /* 1: size the forward for stream_step_fwd_dpo (2 x max_tokens rows) */
  uint64_t cap_bytes;      /* device-memory cap for the workspace; 0 = none           */
} ls_config;

typedef struct ls_ctx ls_ctx;

/* Pre-flight plan: the device workspace (bytes) a context with this config needs.
 * Returns LS_ERR_CAP when that exceeds cfg->cap_bytes (the refusal of a run that
 * will not fit: Soup: Fine-Tune an 8B Model on a 4 GB GPU, "A Practical Quick
 * Start"), LS_ERR_ARG for an unsupported shape. */
int ls_plan(const ls_config* cfg, uint64_t* device_bytes);

/* Create a context.  d_workspace: caller-owned device memory of at least the
 * planned size, 256-byte aligned, kept until ls_destroy.  compute_stream and
 * copy_stream: caller-owned cudaStream_t values (distinct streams).  */
int ls_create(const ls_config* cfg, void* d_workspace, uint64_t ws_bytes, void* compute_stream,
              void* copy_stream, ls_ctx** out);
int ls_destroy(ls_ctx* ctx);

/* Message of the last error on ctx (ctx NULL: the last error of any call on this
 * thread).  Valid until the next call on the same context. */
const char* ls_last_error(const ls_ctx* ctx);

/* NF4-quantise a row-major fp32 matrix [rows, cols] (cols % 64 == 0), on the host:
 * per 64-element block absmax = max|w| (fp32); code = index of the NF4 value nearest
 * to w / absmax (fp32 quotient and distances, ties to the lower index; an all-zero
 * block gets code 7); two codes per byte, element 2i in the high nibble.  Outputs:
 * packed [rows, cols/2] bytes, absmax [rows, cols/64] fp32.  nthreads <= 0: all cores.
 * The 16 code values are QLoRA's NormalFloat-4 table (Dettmers et al. 2023). */
int nf4_quantize(const float* h_w, int64_t rows, int64_t cols, uint8_t* h_packed, float* h_absmax,
                 int32_t nthreads);

/* One NF4 matrix in pinned host memory (cudaHostAlloc or cudaHostRegister). */
typedef struct ls_nf4_host {
  const uint8_t* packed;   /* [rows, cols/2]   */
  const float* absmax;     /* [rows, cols/64]  */
} ls_nf4_host;

/* The frozen weights of one decoder layer, shapes in nn.Linear order [out, in]:
 * q [nh*hd, H], k and v [kv*hd, H], o [H, nh*hd], gate and up [I, H], down [H, I];
 * RMSNorm weights bf16 [H]. */
typedef struct ls_layer_host {
  ls_nf4_host q, k, v, o, gate, up, down;
  const uint16_t* attn_norm;
  const uint16_t* mlp_norm;
} ls_layer_host;

typedef struct ls_vocab_host {
  ls_nf4_host embed;          /* [V, H]; read row by row in place (mapped pinned memory) */
  ls_nf4_host lm_head;        /* [V, H]; ignored when cfg.tied                           */
  const uint16_t* final_norm; /* bf16 [H]                                                */
} ls_vocab_host;

/* Byte offsets of the 16 components inside one layer's slot image, in this order:
 * packed q, k, v, o, gate, up, down; absmax q, k, v, o, gate, up, down; attn_norm,
 * mlp_norm.  A caller that lays out its pinned host copy of a layer the same way
 * (one buffer of image_bytes) gets a single host-to-device copy per layer read. */
int ls_layer_layout(const ls_config* cfg, uint64_t* offsets16, uint64_t* image_bytes);

/* Register a layer's pinned host weights (0 <= layer < L).  Nothing is copied yet;
 * the memory must stay valid and pinned until ls_destroy.  Unpinned memory gives
 * LS_ERR_ARG.  The layer is copied to a device slot each time a pass needs it. */
int load_layer_nf4(ls_ctx* ctx, int32_t layer, const ls_layer_host* h_layer);

/* File-backed layers (the pages' `stream_source` tier: the base on NVMe when host RAM
 * is short; Soup: Fine-Tune an 8B Model on a 4 GB GPU, "The Core Idea: Layer
 * Streaming" and the soup.yaml listing; evermx.com summary).  The layer's slot image
 * (ls_layer_layout) starts at byte `offset` of the file at `path`.  Each time a pass
 * needs the layer it is read on the host (pread; O_DIRECT, bypassing the page cache,
 * when the file system allows it and offset is 4 KiB-aligned) into the next pinned
 * staging buffer, then copied to the slot like a RAM-backed layer, one item ahead of
 * the compute that needs it.  The file must stay unchanged until ls_destroy; results
 * are bit-identical to the same image held in pinned RAM.  Needs ls_set_staging. */
int load_layer_file(ls_ctx* ctx, int32_t layer, const char* path, uint64_t offset);

/* Staging for file-backed layers: nbuf (2..16) caller-owned pinned host buffers of
 * bytes_each (>= the layer image rounded up to 4 KiB, a multiple of 4 KiB), at
 * h_pinned (4 KiB-aligned, consecutive), kept until ls_destroy. */
int ls_set_staging(ls_ctx* ctx, void* h_pinned, uint64_t bytes_each, int32_t nbuf);

/* Register the embedding, vocabulary head and final norm (same rules as above).
 * The final-norm weight is copied to the device here. */
int load_vocab_nf4(ls_ctx* ctx, const ls_vocab_host* h_vocab);

/* Bind the LoRA adapter of one layer (device pointers, caller-owned, kept until the
 * next bind or ls_destroy): A_q [r, H], B_q [nh*hd, r], A_v [r, H], B_v [kv*hd, r]
 * bf16; gradient buffers of the same shapes in fp32, accumulated (+=) by
 * stream_step_bwd.  A layer without an adapter runs the base only. */
int ls_set_adapter(ls_ctx* ctx, int32_t layer, const uint16_t* d_a_q, const uint16_t* d_b_q,
                   const uint16_t* d_a_v, const uint16_t* d_b_v, float* d_g_a_q, float* d_g_b_q,
                   float* d_g_a_v, float* d_g_b_v);

/* Streamed forward pass over T tokens in nseq sequences (d_seq_offsets [nseq+1]
 * cumulative starts, d_tokens int32 [T]).  Writes, per sequence, the sum of the
 * next-token logprobs at the positions d_loss_mask (uint8 [T]) selects into
 * d_seq_logprob_sums [nseq] (fp32).  adapter_on = 0 runs the frozen base alone (the
 * DPO reference pass).  save_acts = 1 keeps the activation store (each layer's
 * input) for stream_step_bwd; the token, offset and mask buffers must then stay
 * valid until that backward. */
int stream_step_fwd(ls_ctx* ctx, const int32_t* d_tokens, int32_t T, int32_t nseq,
                    const int32_t* d_seq_offsets, const uint8_t* d_loss_mask, int32_t adapter_on,
                    int32_t save_acts, float* d_seq_logprob_sums);

/* Shared-read DPO forward: the policy pass (adapter on, activation store kept for
 * stream_step_bwd) and the reference pass (adapter off) over the same T tokens in
 * ONE sweep of the streamed layers.  Each layer is copied to its slot once and
 * serves both passes, which run as one batch of 2T rows (rows 0..T-1 with the
 * adapter, rows T..2T-1 without), so a DPO step reads every layer twice (forward,
 * backward) instead of three times.  The reference logprobs still come from the
 * same streamed base with the adapter off, as in the two-pass form (Show HN:
 * Fine-tune an 8B model on a 4 GB laptop GPU, opening paragraph); every row is
 * computed by the same row-independent kernels.  Writes the policy and reference
 * sequence sums (fp32 [nseq] each; the mask selects positions as in
 * stream_step_fwd).  Needs cfg.dpo_shared_read = 1 (LS_ERR_STATE otherwise).
 * Afterwards seq_logprobs returns 2T values: policy rows, then reference rows. */
int stream_step_fwd_dpo(ls_ctx* ctx, const int32_t* d_tokens, int32_t T, int32_t nseq, const int32_t* d_seq_offsets,
                        const uint8_t* d_loss_mask, float* d_pi_sums, float* d_ref_sums);

/* Per-token logprob log p(token[t+1] | tokens <= t) and log-sum-exp of the last
 * forward pass (fp32 [T] each, [2T] after stream_step_fwd_dpo; 0 logprob at a
 * sequence's last position).  Either output may be NULL. */
int seq_logprobs(ls_ctx* ctx, float* d_token_logprobs, float* d_token_lse);

/* DPO loss over npairs (chosen, rejected) sequence pairs laid out pairwise:
 * z = beta ((pi_c - ref_c) - (pi_r - ref_r)), loss = mean softplus(-z) (=
 * -log sigmoid(z)); d_coeffs [2 npairs] = dL/d(sequence logprob sum) for the
 * backward.  d_pi/d_ref: the policy / reference sums from stream_step_fwd. */
int dpo_loss(ls_ctx* ctx, const float* d_pi, const float* d_ref, int32_t npairs, float beta, float* d_loss,
             float* d_coeffs);

/* SFT loss = -(sum of sequence sums) / count (count = masked positions), and the
 * per-sequence coefficients -1/count for the backward. */
int sft_loss(ls_ctx* ctx, const float* d_seq_sums, int32_t nseq, float count, float* d_loss,
             float* d_coeffs);

/* Reference-free preference losses over npairs (chosen, rejected) pairs laid out
 * pairwise, from the policy sequence sums d_pi [2 npairs] of stream_step_fwd; the
 * response lengths |y| are the counts of selected positions of d_loss_mask in each
 * sequence (d_seq_offsets [2 npairs + 1]).  The pages list SimPO and ORPO among the
 * methods run over the streamed base (axbrief.com, "The Architecture of Low-VRAM
 * Alignment"; evermx.com summary); the formulas are the methods' own:
 *  SimPO (Meng et al. 2024): loss = mean softplus(-(beta (pi_c/|c| - pi_r/|r|) - gamma));
 *  ORPO (Hong et al. 2024): loss = mean [ -pi_c/|c| + lambda softplus(-(lo_c - lo_r)) ],
 *    lo = l - log(1 - e^l) the log odds of the mean logprob l = pi/|y|.
 * d_loss [1]; d_coeffs [2 npairs] = dL/d(sequence sum) for stream_step_bwd.  Neither
 * needs a reference pass. */
int simpo_loss(ls_ctx* ctx, const float* d_pi, const int32_t* d_seq_offsets, const uint8_t* d_loss_mask,
               int32_t npairs, float beta, float gamma, float* d_loss, float* d_coeffs);
int orpo_loss(ls_ctx* ctx, const float* d_pi, const int32_t* d_seq_offsets, const uint8_t* d_loss_mask,
              int32_t npairs, float lambda, float* d_loss, float* d_coeffs);

/* KTO (Ethayarajh et al. 2024; listed on the pages beside DPO) over nseq labelled
 * sequences: r = pi - ref, reference point z0 = max(0, mean r) (held constant for the
 * gradient), loss = mean of lambda_d (1 - sigmoid(beta (r - z0))) over desirable and
 * lambda_u (1 - sigmoid(beta (z0 - r))) over undesirable sequences.  d_desirable
 * uint8 [nseq] (NULL: pair data, even sequences desirable).  d_coeffs [nseq]. */
int kto_loss(ls_ctx* ctx, const float* d_pi, const float* d_ref, const uint8_t* d_desirable, int32_t nseq,
             float beta, float lambda_d, float lambda_u, float* d_loss, float* d_coeffs);

/* Streamed backward of the last saved forward: vocabulary head chunks, then layers
 * L-1..0, each re-streamed and recomputed from its stored input.  d_seq_coeffs
 * [nseq]: dL/d(sequence logprob sum).  LoRA gradients are added (+=) into the bound
 * buffers; the frozen base gets none. */
int stream_step_bwd(ls_ctx* ctx, const float* d_seq_coeffs);

/* Gather every bound LoRA gradient into d_flat_out (fp32, may be NULL), layer by
 * layer in the order A_q, B_q, A_v, B_v, then zero the bound buffers if zero_after. */
int lora_grads(ls_ctx* ctx, float* d_flat_out, int32_t zero_after);

/* fp32 copy of every bound adapter tensor into d_flat_out, in lora_grads' order (the
 * optimizer's master weights before its first step). */
int lora_params(ls_ctx* ctx, float* d_flat_out);

/* AdamW step on every bound adapter (the pages only say the optimizer is picked
 * automatically, "Beyond Streaming" of Soup: Fine-Tune an 8B Model on a 4 GB GPU; this
 * is the usual LoRA choice, Loshchilov & Hutter 2019): with g the bound fp32 gradient,
 *   w = w (1 - lr wd);  m = b1 m + (1-b1) g;  v = b2 v + (1-b2) g^2;
 *   w -= lr (m / (1-b1^t)) / (sqrt(v / (1-b2^t)) + eps)
 * on fp32 master weights d_master, moments d_m, d_v (caller-owned, lora_grads' flat
 * order; d_master from lora_params, d_m = d_v = 0 before step t = 1), then writes
 * bf16(w) into the bound A/B buffers.  zero_grads = 1 clears the gradient buffers. */
int lora_adamw(ls_ctx* ctx, float* d_master, float* d_m, float* d_v, int32_t step, float lr, float beta1,
               float beta2, float eps, float weight_decay, int32_t zero_grads);

/* Wait for the context's streams with a host-side time limit (ms; <= 0: no limit).
 * LS_ERR_TIMEOUT when the limit passes first; LS_ERR_DEVICE when a kernel raised
 * the device error flag. */
int ls_sync(ls_ctx* ctx, int32_t timeout_ms);

typedef struct ls_stats_t {
  uint64_t layer_reads;    /* slot loads of decoder layers over the host link        */
  uint64_t vocab_reads;    /* slot loads of vocabulary-head chunks                    */
  uint64_t h2d_bytes;      /* bytes copied host -> device into slots                  */
  uint64_t slot_reuses;    /* items found already resident in a slot (no copy)        */
  uint64_t workspace_bytes;/* planned device workspace                                */
  uint64_t slot_bytes;     /* one slot                                                */
  uint64_t act_store_bytes;/* activation store                                        */
  int32_t vocab_chunks;
  int32_t vocab_chunk_rows;
  uint64_t kernel_launches; /* kernels this context enqueued                         */
  uint64_t file_bytes;      /* layer-image bytes read from files (load_layer_file)     */
  double file_read_ms;      /* host time spent in those reads                          */
} ls_stats_t;

/* Counters since ls_create (or the last reset). */
int ls_stats(ls_ctx* ctx, ls_stats_t* out, int32_t reset);

/* Kernel classes of the per-launch timing below. */
enum { LS_K_GEMM_FWD = 0, LS_K_GEMM_DX = 1, LS_K_ATTN_FWD = 2, LS_K_ATTN_BWD = 3, LS_K_OTHER = 4, LS_K_CLASSES = 5 };

typedef struct ls_profile_t {
  uint64_t launches[LS_K_CLASSES];
  double ms[LS_K_CLASSES];     /* summed CUDA-event durations on the compute stream       */
  double flop[LS_K_CLASSES];   /* algorithmic FLOPs (2 M N K per matrix product)          */
  double bytes[LS_K_CLASSES];  /* algorithmic bytes (operands read once, outputs written) */
} ls_profile_t;

/* Start (enable = 1, counters reset) or stop (0) timing every kernel this context
 * launches with a pair of CUDA events on the compute stream (up to 65536 launches). */
int ls_profile(ls_ctx* ctx, int32_t enable);

/* Wait for the compute stream and total the timed launches by class. */
int ls_profile_read(ls_ctx* ctx, ls_profile_t* out);

/* Copy entry `layer` of the activation store of the last forward pass run with
 * save_acts = 1 into d_out (bf16 [T, H], caller-owned device memory), on the compute
 * stream: layer 0 is the embedding output (the input of decoder layer 0), layer l
 * the input of decoder layer l, layer L the output of the last decoder layer.  An
 * inspection hook (layer-by-layer checks against a reference implementation); a
 * training step never needs it.  LS_ERR_STATE without a saved forward. */
int ls_read_activation(ls_ctx* ctx, int32_t layer, uint16_t* d_out);

/* Inspection hook for the shared-read DPO forward (the activation store keeps only the
 * policy rows).  With d_buf non-NULL, every later stream_step_fwd_dpo of T tokens also
 * copies the reference rows (adapter off) of each activation-store entry 0..L into
 * d_buf: bf16 [(L+1), T, H], entry l at element offset l * T * H, in the meaning of
 * ls_read_activation (entry 0 the embedding output, entry L the last layer's output).
 * The copies are enqueued on the compute stream after each layer; the step's results
 * are unchanged.  d_buf: caller-owned device memory, 16-byte aligned, at least
 * (L+1) * max_tokens * H * 2 bytes (LS_ERR_ARG otherwise), kept valid until switched
 * off with d_buf = NULL or ls_destroy.  LS_ERR_STATE without cfg.dpo_shared_read.
 * Lets a layer-by-layer check against a reference implementation recompute the very
 * sweep whose loss it grades; a training step never needs it. */
int ls_capture_reference(ls_ctx* ctx, uint16_t* d_buf, uint64_t bytes);

/* Test hook: make every later slot copy on the copy stream first wait host_delay_ms
 * on the host (a host callback), so a bounded ls_sync can be shown to give up.  No
 * GPU fault is involved.  0 switches it off. */
int ls_debug_copy_delay(ls_ctx* ctx, int32_t host_delay_ms);

#ifdef __cplusplus
}
#endif
#endif /* LS_H_ */
