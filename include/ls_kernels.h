/* ls_kernels.h — kernel-level C ABI of libls.so: each hot-path kernel of one
 * streamed training step, callable on its own (parity tests, custom schedules).
 *
 * Every call enqueues device work on `stream` (a cudaStream_t passed as void*) and
 * returns LS_OK or a negative LS_ERR_* status (codes from ls.h); argument errors are
 * caught on the host before any launch.  All pointers are device pointers to
 * caller-owned memory unless named h_*.  bf16 travels as uint16_t; matrices are
 * dense row-major with the given leading dimension (elements).  Shapes: T tokens,
 * H hidden, NF4 matrices W [N, K] in nn.Linear order with K % 64 == 0.
 *
 * Alignment: the kernels move whole 4-, 8- and 16-byte words.  Unless a call says
 * otherwise, bf16 matrices and packed NF4 codes are 16-byte aligned, fp32 matrices
 * 16-byte aligned, absmax and index arrays 4-byte aligned; the narrower cases are
 * listed per call (rmsnorm and SwiGLU backward: bf16 operands 8-byte; LoRA down / du
 * inputs 4-byte; embedding and dequant codes 4-byte; RoPE takes any alignment).
 * A pointer below its call's alignment is refused with LS_ERR_ARG before anything is
 * launched.  Allocations from cudaMalloc or PyTorch are 256-byte aligned.
 */
#ifndef LS_KERNELS_H_
#define LS_KERNELS_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* NF4 dequantisation to bf16: out[r, c] = bf16_rne(q[code] * absmax[r, c/64]) with
 * one fp32 multiply (QLoRA's NormalFloat-4 table; Soup: Fine-Tune an 8B Model on a
 * 4 GB GPU, "The Core Idea: Layer Streaming", "quantization: 4bit # NF4").
 * packed [rows, cols/2], absmax [rows, cols/64], out [rows, cols]. */
int lsk_nf4_dequant(const uint8_t* packed, const float* absmax, int64_t rows, int32_t cols, uint16_t* out,
                    void* stream);

/* NF4-dequant-fused matrix product on the tcgen05 tensor cores (fp32 accumulation).
 *  mode 0 (forward):  out[M, N] = A[M, K] . deq(W)^T            W [N, K]
 *  mode 1 (input grad): out[M, K] = A[M, N] . deq(W)            W [N, K]
 * A: bf16, row pitch lda (multiple of 8); the reduction length must be a multiple
 * of 64.  Optional LoRA extra stage (ext_k = 16 or 32, else 0): ext_a bf16 [M, 64]
 * and ext_b bf16 [out_cols, 64], adding ext_a[:, :ext_k] . ext_b[:, :ext_k]^T into
 * the same accumulator.  epi 0: bf16 out (+ residual bf16 [M, out_cols] when given,
 * added before the one rounding); epi 1: fp32 out; epi 2: fp32 out +=.  ldo, ldr:
 * row pitches of out / residual.  force_bn (0, 128, 256), force_nacc (0, 1, 2) pin
 * the tile shape (0 = automatic). */
int lsk_nf4_gemm(int32_t mode, const uint16_t* A, int64_t lda, int32_t M, const uint8_t* w_packed,
                 const float* w_absmax, int32_t N, int32_t K, const uint16_t* ext_a, const uint16_t* ext_b,
                 int32_t ext_k, int32_t epi, void* out, int64_t ldo, const uint16_t* residual, int64_t ldr,
                 int32_t force_bn, int32_t force_nacc, void* stream);

/* The same product with a stream-K tile schedule available (the stack's own GEMMs use
 * it).  One CTA per SM: whole 256 x 256 tiles round-robin, then the k-iterations of the
 * remaining tiles split evenly over the SMs; a CTA whose share starts inside a tile
 * leaves an fp32 partial in `workspace`, and the CTA holding that tile's first
 * k-iteration adds the partials, in CTA order, before the epilogue (so the result is
 * deterministic, but split tiles sum in a different order than whole ones).  The split
 * launch is cooperative (all CTAs resident at once); its waits are time-bounded and a
 * timeout sets the device error word (lsk_device_error).
 *  split: 0 = the cost model chooses between whole tiles and the split schedule,
 *         1 = split schedule whenever M > 128 (tests), -1 = whole tiles only.
 *  pair_rows: 0, or (with M = 2 pair_rows) a batch of two halves whose identical rows
 *         must give identical outputs: a split tile then takes row r and row
 *         pair_rows + r in its two accumulators, so both meet the same k-splits (whole
 *         tiles sum every row in k order and need no pairing).  Otherwise whole tiles.
 *  workspace: device memory, >= lsk_nf4_gemm_workspace_bytes() bytes, 256-byte
 *         aligned, zero-filled once before its first use (it holds epoch words that
 *         must not match a future launch; no reset is needed between calls).  Calls
 *         sharing a workspace must be ordered (one stream, or events): two in flight at
 *         once corrupt each other's partials.
 * Other arguments and errors as lsk_nf4_gemm. */
uint64_t lsk_nf4_gemm_workspace_bytes(void);

/* The tile shape and schedule lsk_nf4_gemm_sk (and the stack) would launch for a product
 * (host only: no device work, no GPU needed).  Arguments as lsk_nf4_gemm_sk, plus
 * with_workspace (0: no split scratch, whole tiles only) and sms (SMs to plan for;
 * 0 = the current device's, at most 148).  Output tiles are (128 nacc) x bn;
 * ctas = CTAs launched; each first takes whole_per_cta whole tiles round-robin, then an
 * even share of split_iters k-iterations of the remaining tiles (0: none); k_iters =
 * k-iterations of one tile (reduction / 64, + 1 with the LoRA stage); pair_rows = the
 * pairing in effect (tiles_m then counts 128-row blocks of one half). */
typedef struct lsk_gemm_plan {
  int32_t nacc, bn, tiles_m, tiles_n, ctas, whole_per_cta, k_iters, pair_rows;
  int64_t split_iters;
} lsk_gemm_plan;
int lsk_nf4_gemm_plan(int32_t mode, int32_t M, int32_t N, int32_t K, int32_t ext_k, int32_t split,
                      int32_t pair_rows, int32_t with_workspace, int32_t force_bn, int32_t force_nacc, int32_t sms,
                      lsk_gemm_plan* out);
int lsk_nf4_gemm_sk(int32_t mode, const uint16_t* A, int64_t lda, int32_t M, const uint8_t* w_packed,
                    const float* w_absmax, int32_t N, int32_t K, const uint16_t* ext_a, const uint16_t* ext_b,
                    int32_t ext_k, int32_t epi, void* out, int64_t ldo, const uint16_t* residual, int64_t ldr,
                    int32_t force_bn, int32_t force_nacc, int32_t split, int32_t pair_rows, void* workspace,
                    uint64_t workspace_bytes, void* stream);

/* RMSNorm: y = bf16(w * bf16(x * rstd)), rstd = 1/sqrt(mean(x^2) + eps) (fp32).
 * x, y bf16 [T, H] (H % 8 == 0), w bf16 [H], rstd fp32 [T] (may be NULL). */
int lsk_rmsnorm_fwd(const uint16_t* x, const uint16_t* w, uint16_t* y, float* rstd, int32_t T, int32_t H,
                    float eps, void* stream);

/* RMSNorm input gradient: dx (+)= rstd (g - n mean(g n)), g = dy w, n = x rstd.
 * dy, dx fp32 [T, H]; optional dx_bf16 receives bf16(dx) after the update. */
int lsk_rmsnorm_bwd(const float* dy, const uint16_t* x, const float* rstd, const uint16_t* w, float* dx,
                    uint16_t* dx_bf16, int32_t T, int32_t H, int32_t accumulate, void* stream);

/* Host: RoPE tables cos/sin [max_pos, hd/2] for angle p * theta^(-2i/hd) (computed
 * in double, stored fp32). */
int ls_rope_table(float* h_cos, float* h_sin, int32_t max_pos, int32_t head_dim, float theta);

/* Rotate-half RoPE in place on heads 0..nheads-1 of qkv [T, ld] bf16 (pair (i,
 * i+hd/2)), positions pos int32 [T] (each < table rows). */
int lsk_rope_fwd(uint16_t* qkv, int64_t ld, const int32_t* pos, const float* cos_tab, const float* sin_tab,
                 int32_t T, int32_t nheads, int32_t head_dim, void* stream);

/* RoPE backward on an fp32 gradient g [T, ld] (heads 0..nrot_heads-1 rotated back,
 * columns up to ncols copied) written as bf16 into out [T, ld]. */
int lsk_rope_bwd_cast(const float* g, uint16_t* out, int64_t ld, const int32_t* pos, const float* cos_tab,
                      const float* sin_tab, int32_t T, int32_t nrot_heads, int32_t head_dim, int32_t ncols,
                      void* stream);

/* Causal GQA attention forward.  qkv bf16 [T, ld] holds q heads (nh*hd columns),
 * then k heads, then v heads (kv*hd each); sequences by cu int32 [nseq+1];
 * max_len = longest sequence.  out bf16 [T, ldo] (nh*hd columns); lse fp32 [nh, T].
 * qkv and out 16-byte aligned, ld >= (nh + 2 nkv) head_dim and ldo >= nh head_dim, both
 * multiples of 8, 1 <= nseq <= 65535, ceil(max_len / 128) <= 65535 (else LS_ERR_ARG).
 * max_len must not be below any sequence's length (cu lives on the device and is not
 * checked): query tiles past ceil(max_len / 128) are not computed. */
int lsk_attn_fwd(const uint16_t* qkv, int64_t ld, const int32_t* cu, int32_t nseq, int32_t max_len, int32_t nh,
                 int32_t nkv, int32_t head_dim, uint16_t* out, int64_t ldo, float* lse, int32_t T, void* stream);

/* Causal GQA attention backward: from dout bf16 [T, lddo] and the forward's out and
 * lse, writes dq, dk, dv (fp32) into the q/k/v columns of dqkv [T, ldg].
 * d_scratch: fp32 [nh, T].  part: NULL, or fp32 scratch of (nh / nkv) * T * 2 * nkv *
 * head_dim floats (16-byte aligned): dk / dv are then computed per query head by separate
 * CTAs and summed in head order by a second kernel (more CTAs in flight; the same result
 * to fp32 reassociation, and deterministic either way).  qkv, dout, out and dqkv 16-byte
 * aligned; ld and ldg >= (nh + 2 nkv) head_dim, lddo >= nh head_dim; ld, lddo multiples of
 * 8, ldg of 4; nseq and max_len as for lsk_attn_fwd (else LS_ERR_ARG). */
int lsk_attn_bwd(const uint16_t* qkv, int64_t ld, const uint16_t* dout, const uint16_t* out, int64_t lddo,
                 const float* lse, const int32_t* cu, int32_t nseq, int32_t max_len, int32_t nh, int32_t nkv,
                 int32_t head_dim, float* d_scratch, float* dqkv, int64_t ldg, int32_t T, float* part,
                 void* stream);

/* SwiGLU: h = bf16(silu(gate) * up) with gu = [gate | up] bf16 [T, 2I]; backward
 * from dh fp32 [T, I] to dgu bf16 [T, 2I]. */
int lsk_swiglu_fwd(const uint16_t* gu, uint16_t* h, int32_t T, int32_t I, void* stream);
int lsk_swiglu_bwd(const float* dh, const uint16_t* gu, uint16_t* dgu, int32_t T, int32_t I, void* stream);

/* LoRA down-projection for the forward extra stage: u_ext bf16 [T, 64] =
 * [bf16(s x A_q^T) | bf16(s x A_v^T) | 0]; x bf16 [T, ldx], A bf16 [r, K] (either
 * may be NULL), r <= 16 (Soup: Fine-Tune an 8B Model on a 4 GB GPU, soup.yaml
 * listing: r 16 on q_proj, v_proj).  K a multiple of 16, ldx even. */
int lsk_lora_down(const uint16_t* x, int64_t ldx, const uint16_t* a_q, const uint16_t* a_v, int32_t r,
                  int32_t K, float s, uint16_t* u_ext, int32_t T, void* stream);

/* du fp32 [T, 32] = s [dY_q B_q | dY_v B_v] (dY columns at col_q / col_v of dy
 * [T, ldy]) and its bf16 copy du_ext [T, 64] (columns 32..63 zero).  ldy, col_q and
 * col_v even; nq, nv multiples of 16.  Both down-projections run on the tensor cores
 * (mma.sync, fp32 accumulation) with a fixed-order reduction over K. */
int lsk_lora_du(const uint16_t* dy, int64_t ldy, int32_t col_q, int32_t nq, const uint16_t* b_q,
                int32_t col_v, int32_t nv, const uint16_t* b_v, int32_t r, float s, float* du, uint16_t* du_ext,
                int32_t T, void* stream);

/* Deterministic outer product over tokens: out (+)= X^T U with X bf16 [T, ldx]
 * (ncols columns) and U (fp32 u_f32 or bf16 u_bf16, [T, ldu], first r columns; only
 * those r columns are read, so a compact U with ldu = r is fine).
 * layout 0: out [ncols, r] (dB shape); layout 1: out [r, ncols] (dA shape).
 * X rows must be 16-byte aligned (X 16-byte aligned, ldx and ncols multiples of 8);
 * ldx >= ncols, ldu >= r, ceil(T / rows_per_chunk) <= 65535, else LS_ERR_ARG.
 * scratch fp32 of nchunks * ncols * 16 floats, nchunks = ceil(T / rows_per_chunk). */
int lsk_lora_outer(const uint16_t* X, int64_t ldx, int32_t ncols, const float* u_f32, const uint16_t* u_bf16,
                   int32_t ldu, int32_t r, int32_t T, int32_t layout, int32_t accumulate, float* scratch,
                   int32_t rows_per_chunk, float* out, void* stream);

/* Size (fp32 elements) of the fixed scratch of lsk_lora_outer_noalloc: 2^21 floats
 * (8 MiB).  A call needs ceil(T / rows_per_chunk) * ncols * 16 of them. */
#define LS_OUTER_NOALLOC_SCRATCH_FLOATS 2097152

/* lsk_lora_outer for callers that cannot allocate device memory: the same
 * deterministic outer product over tokens (same arguments minus `scratch`, same
 * result bit for bit), with its partial sums kept in a fixed array inside the
 * library instead of caller scratch.  Meant for code that runs where cudaMalloc is
 * off limits -- inside a host framework whose memory pool owns all device memory,
 * or on a path that must not take cudaMalloc's implicit device synchronisation.  The
 * Soup pages have no counterpart; this is a library-usage convenience.
 *  - The array (LS_OUTER_NOALLOC_SCRATCH_FLOATS floats) is part of the library image:
 *    every GPU that loads the library holds it until the process exits.
 *  - The first call on a device looks the array's device address up (with that
 *    device current) and caches it; make that first call before any stream capture.
 *    The cached address belongs to the device's primary context: after a
 *    cudaDeviceReset on that device it is stale, so do not call this again in the
 *    same process after such a reset.
 *  - Every call on a device shares the one array and it keeps the last call's
 *    contents; each call writes every element it later reads, so nothing needs
 *    clearing.  Calls whose kernels overlap on the GPU (e.g. on two streams) race on
 *    the array: serialise them.
 *  - Sizes beyond the array (ceil(T / rows_per_chunk) * ncols * 16 floats) return
 *    LS_ERR_ARG with a message; nothing is launched.  No call allocates or frees
 *    device memory. */
int lsk_lora_outer_noalloc(const uint16_t* X, int64_t ldx, int32_t ncols, const float* u_f32, const uint16_t* u_bf16,
                           int32_t ldu, int32_t r, int32_t T, int32_t layout, int32_t accumulate,
                           int32_t rows_per_chunk, float* out, void* stream);

/* Extra-stage operands built from the adapter: B_ext [N, 64] (q rows [q0, q0+nq)
 * take B_q in columns 0..r-1, v rows [v0, v0+nv) take B_v in columns 16..16+r-1)
 * and A_ext [K, 64] (row k = [A_q[:, k] | A_v[:, k] | 0]). */
int lsk_build_ext_fwd(const uint16_t* b_q, int32_t q0, int32_t nq, const uint16_t* b_v, int32_t v0, int32_t nv,
                      int32_t r, int32_t N, uint16_t* ext, void* stream);
int lsk_build_ext_bwd(const uint16_t* a_q, const uint16_t* a_v, int32_t r, int32_t K, uint16_t* ext,
                      void* stream);

/* NF4 embedding gather: x[t] = dequant(row tokens[t]) of the V-row table; packed/absmax
 * may be mapped pinned host memory.  A token id outside [0, V) gives a zero row and sets
 * the device error word (lsk_device_error). */
int lsk_embed_gather(const int32_t* tokens, const uint8_t* packed, const float* absmax, int32_t V, uint16_t* x,
                     int32_t T, int32_t H, void* stream);

/* Vocabulary logprobs without materialising the logits: logits = h . deq(W)^T
 * (h bf16 [T, H], W NF4 [V, H]) reduced on the fly to per-128-column (max, sum-exp)
 * partials (scratch fp32 2 * T * ceil(V/128)), then lse [T], the target logit, and
 * lp[t] = logit[t, target[t]] - lse[t] (0 where target[t] < 0).  tgt_logit scratch
 * fp32 [T]. */
int lsk_vocab_logprob(const uint16_t* h, int32_t T, int32_t H, const uint8_t* w_packed, const float* w_absmax,
                      int32_t V, const int32_t* targets, float* scratch, float* tgt_logit, float* lse, float* lp,
                      void* stream);

/* Vocabulary backward for one chunk of rows [v0, v0 + n) of W: dlogits bf16
 * [T, n] = coef[t] (onehot(target[t] - v0) - exp(logit - lse[t])), then
 * dh (+)= dlogits . deq(W_chunk) (fp32 [T, H]). */
int lsk_vocab_bwd(const uint16_t* h, int32_t T, int32_t H, const uint8_t* w_packed, const float* w_absmax,
                  int32_t v0, int32_t n, const int32_t* targets, const float* lse, const float* coef,
                  uint16_t* dlogits, float* dh, int32_t accumulate, void* stream);

/* The bounded device wait every cross-CTA handshake of these kernels uses (the split
 * GEMM's partial tiles), on its own: one thread waits until the uint32 at flag equals
 * value or limit_ns nanoseconds (device %globaltimer) have passed, then writes status
 * (int32, device): 0 = seen, 1 = the limit ran out, in which case the device error word
 * (lsk_device_error) is also raised.  The kernel returns either way; the context stays
 * usable.  Lets a caller check the failure path of a wait with a flag nothing sets. */
int lsk_wait_flag(const uint32_t* flag, uint32_t value, int64_t limit_ns, int32_t* status, void* stream);

/* Device error flag raised by kernels whose bounded waits ran out (0 = none). */
int lsk_device_error(int32_t* h_out, int32_t reset);

#ifdef __cplusplus
}
#endif
#endif /* LS_KERNELS_H_ */
