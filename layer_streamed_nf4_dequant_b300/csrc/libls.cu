// libls: layer-streamed NF4 LoRA fine-tuning on one B300 — C ABI implementation.
//
// The frozen base lives in pinned host RAM and is copied one decoder layer at a time
// into one of two device slots on a dedicated copy stream while the other slot's
// layer computes ("The Core Idea: Layer Streaming" and FAQ of Soup: Fine-Tune an 8B
// Model on a 4 GB GPU).  Forward passes store each layer's input (the activation
// store); the backward re-streams layers in reverse and recomputes each from its
// stored input.  DPO's reference pass re-streams the same base with the adapter off
// (Show HN: Fine-tune an 8B model on a 4 GB laptop GPU).  Every kernel is
// deterministic, so a streamed pass equals a resident pass bit for bit.
//
// One translation unit: kernels and host code are compiled together.
#include <algorithm>
#include <chrono>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <functional>
#include <fcntl.h>
#include <unistd.h>
#include <cerrno>
#include <climits>
#include <mutex>
#include <string>
#include <thread>
#include <vector>

#include "common.cuh"
#include "nf4_gemm.cuh"
#include "gemm_host.cuh"
#include "pointwise.cuh"
#include "attention.cuh"
#include "attention_tc.cuh"
#include "ls.h"
#include "ls_kernels.h"

using ls::GemmArgs;
using ls::GemmCall;
typedef __nv_bfloat16 bf16;

namespace {

thread_local std::string g_thread_err;

int set_thread_err(int code, const std::string& m) {
  g_thread_err = m;
  return code;
}

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// A pointer that is given and not a multiple of a bytes (a power of two): the kernels read
// and write whole 4-, 8- or 16-byte words, and a misaligned word access faults.
inline bool misaligned(const void* p, uintptr_t a) { return p && (reinterpret_cast<uintptr_t>(p) & (a - 1)) != 0; }

constexpr int kLoraSplitMax = 8;   // K slices of the LoRA projections (workspace scratch)

// ------------------------------------------------------------------ host NF4 quantiser
// QLoRA's NormalFloat-4 code values (Dettmers et al. 2023, Appendix E).
const float kNF4Host[16] = {-1.0f, -0.6961928009986877f, -0.5250730514526367f, -0.39491748809814453f,
                            -0.28444138169288635f, -0.18477343022823334f, -0.09105003625154495f, 0.0f,
                            0.07958029955625534f, 0.16093020814657211f, 0.24611230194568634f,
                            0.33791524171829224f, 0.44070982933044434f, 0.5626170039176941f,
                            0.7229568362236023f, 1.0f};

void quantize_rows(const float* w, int64_t r0, int64_t r1, int64_t cols, uint8_t* packed, float* absmax) {
  const int64_t nb = cols / 64;
  for (int64_t r = r0; r < r1; ++r) {
    for (int64_t b = 0; b < nb; ++b) {
      const float* blk = w + r * cols + b * 64;
      float a = 0.f;
      for (int i = 0; i < 64; ++i) a = std::max(a, std::fabs(blk[i]));
      absmax[r * nb + b] = a;
      uint8_t* out = packed + r * (cols / 2) + b * 32;
      for (int i = 0; i < 64; i += 2) {
        uint8_t c[2];
        for (int e = 0; e < 2; ++e) {
          if (a == 0.f) {
            c[e] = 7;
            continue;
          }
          const float x = blk[i + e] / a;   // fp32 quotient
          int best = 0;
          float bd = std::fabs(x - kNF4Host[0]);
          for (int j = 1; j < 16; ++j) {
            const float d = std::fabs(x - kNF4Host[j]);
            if (d < bd) {   // strict: ties keep the lower index
              bd = d;
              best = j;
            }
          }
          c[e] = (uint8_t)best;
        }
        out[i / 2] = (uint8_t)((c[0] << 4) | c[1]);
      }
    }
  }
}

}  // namespace

// ====================================================================== context

struct LayerLayout {
  size_t off[16];
  size_t bytes;
};

struct ls_ctx {
  ls_config cfg{};
  cudaStream_t cs = nullptr, cp = nullptr;
  uint8_t* ws = nullptr;
  uint64_t ws_bytes = 0;
  int err = 0;
  std::string msg;

  int L, H, nh, nkv, hd, I, V, r, nq, nkvd, nqkv, Tmax, maxlen;
  LayerLayout lay{};
  size_t slot_bytes = 0;
  int vrows = 0, nvch = 0;
  size_t vch_abs_off = 0;   // absmax offset inside a vocabulary chunk image

  uint8_t* slot[2] = {nullptr, nullptr};
  int slot_item[2] = {-1, -1};
  long long slot_use[2] = {0, 0};
  long long use_clock = 0;
  cudaEvent_t ev_ready[2] = {}, ev_free[2] = {};
  bool free_rec[2] = {false, false};
  std::vector<uint8_t*> res_img;   // resident mode: one image per item
  std::vector<char> res_loaded;

  std::vector<ls_layer_host> hl;
  std::vector<char> hl_ok;
  // file-backed layers (the "NVMe" tier): slot image at byte offset of a file
  struct FileSrc {
    int fd = -1;
    bool direct = false;
    uint64_t off = 0;
  };
  std::vector<FileSrc> lf;
  std::vector<std::pair<std::string, std::pair<int, int>>> files;   // path -> (O_DIRECT fd, buffered fd)
  std::vector<uint8_t*> stage;            // caller's pinned staging buffers
  std::vector<cudaEvent_t> stage_ev;      // H2D copy out of each buffer
  std::vector<char> stage_used;
  size_t stage_bytes = 0;
  int stage_next = 0;
  ls_vocab_host hv{};
  bool hv_ok = false;
  const uint8_t* emb_p = nullptr;   // device-visible pointers to the mapped pinned embedding
  const float* emb_a = nullptr;

  struct Ad {
    const bf16 *aq = nullptr, *bq = nullptr, *av = nullptr, *bv = nullptr;
    float *gaq = nullptr, *gbq = nullptr, *gav = nullptr, *gbv = nullptr;
    bool on = false;
  };
  std::vector<Ad> ad;

  // device buffers (inside the workspace)
  bf16* wf = nullptr;
  float *rope_cos = nullptr, *rope_sin = nullptr;
  bf16 *acts = nullptr, *xping = nullptr;
  bf16 *n1, *qkv, *attn_o, *x1, *n2, *gu, *hbuf, *u_ext, *ext_fwd;
  float *rstd1, *rstd2, *lse_attn;
  float *gx, *dh, *dn, *Dattn, *dqkv_f, *du, *lora_part;
  bf16 *gx_bf, *dgu, *do_bf, *dqkv_bf, *du_ext, *ext_bwd;
  bf16 *hf_save, *hf_tmp, *dlogits;
  float *rstdf_save, *rstdf_tmp, *pmax, *psum, *tgt_logit, *lse_save, *lse_tmp, *lp, *coef, *dhf, *loss_tmp;
  int32_t *tgt, *pos;
  int32_t *tok2 = nullptr, *cu2 = nullptr;   // shared-read DPO forward: doubled batch
  float* attn_part = nullptr;                 // per-query-head dk / dv partials
  ls::SkWorkspace skw;                        // split-tile (stream-K) scratch of the NF4 GEMMs
  int pair_rows = 0;                          // T while the shared-read DPO forward runs
  bf16* ref_cap = nullptr;                    // ls_capture_reference: caller's [(L+1), T, H] buffer
  uint64_t ref_cap_bytes = 0;
  int Tf = 0;                                 // forward row capacity (2 max_tokens with shared read)
  int P = 0;
  size_t lora_part_floats = 0;

  bool saved = false;
  const int32_t* s_tokens = nullptr;
  const int32_t* s_cu = nullptr;
  const uint8_t* s_mask = nullptr;
  int s_T = 0, s_nseq = 0;
  int last_T = 0;
  const float* last_lse = nullptr;

  ls_stats_t st{};
  double file_ms = 0.0;
  uint64_t file_bytes = 0;
  int copy_delay_ms = 0;

  // per-launch CUDA-event timing on the compute stream (ls_profile)
  bool prof_on = false;
  std::vector<cudaEvent_t> prof_ev;
  std::vector<int> prof_cls;
  std::vector<double> prof_flop, prof_bytes;
  size_t prof_used = 0;
};

namespace {

// Split-tile scratch for the stack's NF4 GEMMs.  The shared-read DPO forward stacks the
// policy and reference copies of the batch into one product of 2T rows; marking the
// halves (pair_rows = T) makes identical policy and reference rows round identically
// under any tile schedule (the B = 0 start has policy = reference exactly).
ls::SkWorkspace gemm_ws(const ls_ctx* c) {
  ls::SkWorkspace w = c->skw;
  w.pair_rows = c->pair_rows;
  return w;
}

int fail(ls_ctx* c, int code, const std::string& m) {
  if (c && c->err == 0) {
    c->err = code;
    c->msg = m;
  }
  g_thread_err = m;
  return code;
}

#define CK(call)                                                                              \
  do {                                                                                        \
    cudaError_t e_ = (call);                                                                  \
    if (e_ != cudaSuccess) return fail(c, LS_ERR_CUDA, std::string(#call) + ": " + cudaGetErrorString(e_)); \
  } while (0)

#define CKL()                                                                                 \
  do {                                                                                        \
    cudaError_t e_ = cudaGetLastError();                                                      \
    if (e_ != cudaSuccess) return fail(c, LS_ERR_CUDA, std::string("launch: ") + cudaGetErrorString(e_)); \
  } while (0)

constexpr size_t kProfMax = 1 << 16;

inline void pbeg(ls_ctx* c) {
  if (c->prof_on && c->prof_used < kProfMax) cudaEventRecord(c->prof_ev[2 * c->prof_used], c->cs);
}
inline void pend(ls_ctx* c, int cls, double flop, double bytes) {
  c->st.kernel_launches++;
  if (c->prof_on && c->prof_used < kProfMax) {
    cudaEventRecord(c->prof_ev[2 * c->prof_used + 1], c->cs);
    c->prof_cls[c->prof_used] = cls;
    c->prof_flop[c->prof_used] = flop;
    c->prof_bytes[c->prof_used] = bytes;
    ++c->prof_used;
  }
}

// Time one enqueue (nk kernels) on the compute stream as class `cls`.
#define TIMED(cls, flop, bytes, nk, ...)                                                      \
  do {                                                                                        \
    pbeg(c);                                                                                  \
    __VA_ARGS__;                                                                              \
    cudaError_t e_ = cudaGetLastError();                                                      \
    if (e_ != cudaSuccess) return fail(c, LS_ERR_CUDA, std::string("launch: ") + cudaGetErrorString(e_)); \
    pend(c, cls, flop, bytes);                                                                \
    c->st.kernel_launches += (nk) - 1;                                                        \
  } while (0)

#define GEMM_T(cls, flop, bytes, call)                                                        \
  do {                                                                                        \
    pbeg(c);                                                                                  \
    cudaError_t ge_ = (call);                                                                 \
    if (ge_ != cudaSuccess) return fail(c, LS_ERR_CUDA, std::string("gemm: ") + cudaGetErrorString(ge_)); \
    pend(c, cls, flop, bytes);                                                                \
  } while (0)

// Algorithmic cost of one NF4 matrix product: 2 M N K flops (+ the LoRA stage);
// bytes = activation read once + NF4 weight (0.5625 B per weight) + output (+ residual).
inline double gemm_flop(int mode, int M, int Nw, int Kw, int ext_k) {
  const double Nout = mode == ls::GEMM_FWD ? Nw : Kw;
  return 2.0 * M * (double)Nw * Kw + 2.0 * M * Nout * ext_k;
}
inline double gemm_bytes(int mode, int M, int Nw, int Kw, int out_bytes, bool residual) {
  const double Nout = mode == ls::GEMM_FWD ? Nw : Kw, Kred = mode == ls::GEMM_FWD ? Kw : Nw;
  return 2.0 * M * Kred + 0.5625 * (double)Nw * Kw + (double)M * Nout * (out_bytes + (residual ? 2 : 0));
}

int check_cfg(const ls_config* cfg, std::string& why) {
  if (!cfg) { why = "null config"; return LS_ERR_ARG; }
  const ls_config& k = *cfg;
  if (k.layers < 1 || k.hidden < 64 || k.hidden % 64) { why = "hidden must be a positive multiple of 64"; return LS_ERR_ARG; }
  if (k.heads < 1 || k.kv_heads < 1 || k.heads % k.kv_heads) { why = "heads must be a multiple of kv_heads"; return LS_ERR_ARG; }
  if (k.head_dim != 64 && k.head_dim != 128) { why = "head_dim must be 64 or 128"; return LS_ERR_ARG; }
  if (k.inter < 64 || k.inter % 64) { why = "inter must be a multiple of 64"; return LS_ERR_ARG; }
  if (k.vocab < 64 || k.vocab % 64) { why = "vocab must be a multiple of 64"; return LS_ERR_ARG; }
  if ((k.heads * k.head_dim) % 64 || (k.kv_heads * k.head_dim) % 64) { why = "head widths must be multiples of 64"; return LS_ERR_ARG; }
  if (k.lora_r < 1 || k.lora_r > 16) { why = "lora_r must be in 1..16"; return LS_ERR_ARG; }
  if (k.max_tokens < 1 || k.max_seqs < 1) { why = "max_tokens and max_seqs must be positive"; return LS_ERR_ARG; }
  if (k.vocab_chunk_rows < 0 || k.vocab_chunk_rows % 256) { why = "vocab_chunk_rows must be a multiple of 256"; return LS_ERR_ARG; }
  return LS_OK;
}

LayerLayout layer_layout(const ls_config& k) {
  const size_t H = k.hidden, I = k.inter, nq = (size_t)k.heads * k.head_dim, nkv = (size_t)k.kv_heads * k.head_dim;
  const size_t rows[7] = {nq, nkv, nkv, H, I, I, H};
  const size_t cols[7] = {H, H, H, nq, H, H, I};
  LayerLayout L{};
  size_t o = 0;
  // packed groups: [q k v] [o] [gate up] [down], each group 256-aligned
  const int group_start[7] = {1, 0, 0, 1, 1, 0, 1};
  for (int m = 0; m < 7; ++m) {
    if (group_start[m]) o = align_up(o, 256);
    L.off[m] = o;
    o += rows[m] * cols[m] / 2;
  }
  for (int m = 0; m < 7; ++m) {
    if (group_start[m]) o = align_up(o, 256);
    L.off[7 + m] = o;
    o += rows[m] * (cols[m] / 64) * 4;
  }
  o = align_up(o, 256);
  L.off[14] = o;
  o += H * 2;
  o = align_up(o, 256);
  L.off[15] = o;
  o += H * 2;
  L.bytes = align_up(o, 256);
  return L;
}

struct Planned {
  size_t total = 0;
  size_t slot_bytes = 0, act_bytes = 0;
  int vrows = 0, nvch = 0, P = 0;
  size_t vch_abs_off = 0;
};

// Bump allocation of the workspace.  With base == nullptr only sizes are computed.
struct Bump {
  uint8_t* base;
  size_t off = 0;
  template <class T>
  T* take(size_t count) {
    off = align_up(off, 256);
    T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
    off += count * sizeof(T);
    return p;
  }
};

void vocab_chunking(const ls_config& k, size_t slot_bytes, int& vrows, int& nvch, size_t& abs_off) {
  const size_t H = k.hidden;
  const size_t row_bytes = H / 2 + (H / 64) * 4;
  int rows = k.vocab_chunk_rows;
  if (rows == 0) {
    rows = (int)((slot_bytes - 512) / row_bytes / 256 * 256);
    if (rows < 256) rows = 256;
  }
  if (rows > k.vocab) rows = (k.vocab + 255) / 256 * 256;
  vrows = rows;
  nvch = (k.vocab + rows - 1) / rows;
  abs_off = align_up((size_t)rows * (H / 2), 256);
}

// Lay the whole workspace out (ctx may be null: sizes only).
Planned lay_out(const ls_config& k, ls_ctx* c) {
  Planned p;
  const LayerLayout ll = layer_layout(k);
  const size_t T = k.max_tokens, H = k.hidden, I = k.inter;
  // forward-pass buffers hold 2T rows when the policy and reference passes share a sweep
  const size_t Tf = k.dpo_shared_read ? 2 * T : T;
  const size_t nq = (size_t)k.heads * k.head_dim, nkvd = (size_t)k.kv_heads * k.head_dim, nqkv = nq + 2 * nkvd;
  const int maxlen = k.max_seq_len > 0 ? k.max_seq_len : k.max_tokens;
  size_t slot = ll.bytes;
  int vrows, nvch;
  size_t abs_off;
  vocab_chunking(k, slot, vrows, nvch, abs_off);
  const size_t vimg = abs_off + (size_t)vrows * (H / 64) * 4;
  if (vimg > slot) slot = align_up(vimg, 256);
  p.slot_bytes = slot;
  p.vrows = vrows;
  p.nvch = nvch;
  p.vch_abs_off = abs_off;
  p.P = (k.vocab + 127) / 128;

  Bump b{c ? c->ws : nullptr};
  uint8_t* slots = nullptr;
  if (k.resident) {
    slots = b.take<uint8_t>((size_t)k.layers * ll.bytes + (size_t)nvch * align_up(vimg, 256) + 256);
  } else {
    slots = b.take<uint8_t>(2 * slot);
  }
  bf16* wf = b.take<bf16>(H);
  float* rc = b.take<float>((size_t)maxlen * k.head_dim / 2);
  float* rsn = b.take<float>((size_t)maxlen * k.head_dim / 2);
  const size_t act0 = b.off;
  bf16* acts = b.take<bf16>((size_t)(k.layers + 1) * T * H);
  p.act_bytes = b.off - act0;
  bf16* xping = b.take<bf16>(2 * Tf * H);
  // forward layer scratch
  bf16* n1 = b.take<bf16>(Tf * H);
  bf16* qkv = b.take<bf16>(Tf * nqkv);
  bf16* ao = b.take<bf16>(Tf * nq);
  bf16* x1 = b.take<bf16>(Tf * H);
  bf16* n2 = b.take<bf16>(Tf * H);
  bf16* gu = b.take<bf16>(Tf * 2 * I);
  bf16* hb = b.take<bf16>(Tf * I);
  bf16* uext = b.take<bf16>(Tf * 64);
  bf16* extf = b.take<bf16>(nqkv * 64);
  float* rstd1 = b.take<float>(Tf);
  float* rstd2 = b.take<float>(Tf);
  float* lsea = b.take<float>((size_t)k.heads * Tf);
  // backward
  float* gx = b.take<float>(T * H);
  bf16* gxb = b.take<bf16>(T * H);
  float* dn = b.take<float>(T * H);
  bf16* dob = b.take<bf16>(T * nq);
  float* Da = b.take<float>((size_t)k.heads * T);
  float* dqf = b.take<float>(T * nqkv);
  bf16* dqb = b.take<bf16>(T * nqkv);
  float* du = b.take<float>(T * 32);
  bf16* duext = b.take<bf16>(T * 64);
  bf16* extb = b.take<bf16>(H * 64);
  const int chunks = (int)((T + 127) / 128);
  // LoRA scratch: outer-product partials, and the K-split partials of the projections
  const size_t lpf = std::max((size_t)chunks * std::max(nqkv, H) * 16, (size_t)kLoraSplitMax * T * 32);
  float* lpart = b.take<float>(lpf);
  // attention backward: dk / dv of every query head before the ordered sum over its group
  float* apart = k.heads > k.kv_heads ? b.take<float>((size_t)k.heads / k.kv_heads * T * 2 * nkvd) : nullptr;
  // union: layer-backward big buffers / vocabulary dlogits
  const size_t u0 = align_up(b.off, 256);
  Bump u1{c ? c->ws : nullptr, u0};
  float* dh = u1.take<float>(T * I);
  bf16* dgu = u1.take<bf16>(T * 2 * I);
  Bump u2{c ? c->ws : nullptr, u0};
  bf16* dl = u2.take<bf16>(T * (size_t)vrows);
  b.off = std::max(u1.off, u2.off);
  // vocabulary / loss
  bf16* hfs = b.take<bf16>(T * H);
  bf16* hft = b.take<bf16>(Tf * H);
  float* rfs = b.take<float>(T);
  float* rft = b.take<float>(Tf);
  float* pmax = b.take<float>(Tf * (size_t)p.P);
  float* psum = b.take<float>(Tf * (size_t)p.P);
  float* tl = b.take<float>(Tf);
  float* lses = b.take<float>(T);
  float* lset = b.take<float>(Tf);
  float* lp = b.take<float>(Tf);
  float* coef = b.take<float>(T);
  float* dhf = b.take<float>(T * H);
  float* losst = b.take<float>(64);
  int32_t* tgt = b.take<int32_t>(Tf);
  int32_t* pos = b.take<int32_t>(Tf);
  int32_t* tok2 = k.dpo_shared_read ? b.take<int32_t>(Tf) : nullptr;
  int32_t* cu2 = k.dpo_shared_read ? b.take<int32_t>(2 * (size_t)k.max_seqs + 1) : nullptr;
  uint8_t* skbase = b.take<uint8_t>(ls::kSkWorkspaceBytes);
  p.total = align_up(b.off, 256);

  if (c) {
    c->slot_bytes = slot;
    if (k.resident) {
      c->res_img.resize(k.layers + nvch);
      size_t o = 0;
      for (int i = 0; i < k.layers; ++i) { c->res_img[i] = slots + o; o += ll.bytes; }
      for (int i = 0; i < nvch; ++i) { c->res_img[k.layers + i] = slots + o; o += align_up(vimg, 256); }
      c->res_loaded.assign(k.layers + nvch, 0);
    } else {
      c->slot[0] = slots;
      c->slot[1] = slots + slot;
    }
    c->wf = wf; c->rope_cos = rc; c->rope_sin = rsn; c->acts = acts; c->xping = xping;
    c->n1 = n1; c->qkv = qkv; c->attn_o = ao; c->x1 = x1; c->n2 = n2; c->gu = gu; c->hbuf = hb;
    c->u_ext = uext; c->ext_fwd = extf; c->rstd1 = rstd1; c->rstd2 = rstd2; c->lse_attn = lsea;
    c->gx = gx; c->gx_bf = gxb; c->dn = dn; c->do_bf = dob; c->Dattn = Da; c->dqkv_f = dqf; c->dqkv_bf = dqb;
    c->du = du; c->du_ext = duext; c->ext_bwd = extb; c->lora_part = lpart; c->lora_part_floats = lpf;
    c->dh = dh; c->dgu = dgu; c->dlogits = dl;
    c->hf_save = hfs; c->hf_tmp = hft; c->rstdf_save = rfs; c->rstdf_tmp = rft; c->pmax = pmax; c->psum = psum;
    c->tgt_logit = tl; c->lse_save = lses; c->lse_tmp = lset; c->lp = lp; c->coef = coef; c->dhf = dhf;
    c->loss_tmp = losst; c->tgt = tgt; c->pos = pos; c->P = p.P;
    c->tok2 = tok2; c->cu2 = cu2; c->Tf = (int)Tf; c->attn_part = apart;
    c->skw = ls::sk_workspace_at(skbase);
    c->vrows = vrows; c->nvch = nvch; c->vch_abs_off = abs_off;
  }
  return p;
}

// ------------------------------------------------------------------ kernel launch helpers

inline int grid1d(long long n, int threads, int cap = 148 * 16) {
  long long g = (n + threads - 1) / threads;
  if (g < 1) g = 1;
  if (g > cap) g = cap;
  return (int)g;
}

// RMSNorm launches: one block per row with the row's slice in registers for rows up to
// 8192 wide (the row-per-block kernels), one warp per row beyond that.
template <int V>
void rmsnorm_fwd_v(const bf16* x, const bf16* w, bf16* y, float* rstd, int T, int H, float eps, cudaStream_t st) {
  ls::rmsnorm_fwd_row_kernel<V><<<T, 128, 0, st>>>(x, w, y, rstd, H, eps);
}
cudaError_t rmsnorm_fwd(const bf16* x, const bf16* w, bf16* y, float* rstd, int T, int H, float eps,
                        cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  switch ((H / 8 + 127) / 128) {
    case 1: rmsnorm_fwd_v<1>(x, w, y, rstd, T, H, eps, st); break;
    case 2: rmsnorm_fwd_v<2>(x, w, y, rstd, T, H, eps, st); break;
    case 3: rmsnorm_fwd_v<3>(x, w, y, rstd, T, H, eps, st); break;
    case 4: rmsnorm_fwd_v<4>(x, w, y, rstd, T, H, eps, st); break;
    case 5: rmsnorm_fwd_v<5>(x, w, y, rstd, T, H, eps, st); break;
    case 6: rmsnorm_fwd_v<6>(x, w, y, rstd, T, H, eps, st); break;
    case 7: rmsnorm_fwd_v<7>(x, w, y, rstd, T, H, eps, st); break;
    case 8: rmsnorm_fwd_v<8>(x, w, y, rstd, T, H, eps, st); break;
    default: ls::rmsnorm_fwd_kernel<<<(T + 7) / 8, 256, 0, st>>>(x, w, y, rstd, T, H, eps);
  }
  return cudaGetLastError();
}
template <int V>
void rmsnorm_bwd_v(const float* dy, const bf16* x, const float* rstd, const bf16* w, float* dx, bf16* dxb, int T,
                   int H, int acc, cudaStream_t st) {
  ls::rmsnorm_bwd_row_kernel<V><<<T, 256, 0, st>>>(dy, x, rstd, w, dx, dxb, H, acc);
}
cudaError_t rmsnorm_bwd(const float* dy, const bf16* x, const float* rstd, const bf16* w, float* dx, bf16* dxb, int T,
                        int H, int acc, cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  switch ((H / 4 + 255) / 256) {
    case 1: rmsnorm_bwd_v<1>(dy, x, rstd, w, dx, dxb, T, H, acc, st); break;
    case 2: rmsnorm_bwd_v<2>(dy, x, rstd, w, dx, dxb, T, H, acc, st); break;
    case 3: rmsnorm_bwd_v<3>(dy, x, rstd, w, dx, dxb, T, H, acc, st); break;
    case 4: rmsnorm_bwd_v<4>(dy, x, rstd, w, dx, dxb, T, H, acc, st); break;
    case 5: rmsnorm_bwd_v<5>(dy, x, rstd, w, dx, dxb, T, H, acc, st); break;
    case 6: rmsnorm_bwd_v<6>(dy, x, rstd, w, dx, dxb, T, H, acc, st); break;
    case 7: rmsnorm_bwd_v<7>(dy, x, rstd, w, dx, dxb, T, H, acc, st); break;
    case 8: rmsnorm_bwd_v<8>(dy, x, rstd, w, dx, dxb, T, H, acc, st); break;
    default: ls::rmsnorm_bwd_kernel<<<(T + 7) / 8, 256, 0, st>>>(dy, x, rstd, w, dx, dxb, T, H, acc);
  }
  return cudaGetLastError();
}

// RoPE launches: the 16-byte kernels when rows and pointers allow 16-byte access.
inline bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }
cudaError_t rope_fwd(bf16* qkv, long long ld, const int* pos, const float* ct, const float* stt, int T, int nheads,
                     int hd, cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  if (ld % 8 == 0 && al16(qkv) && al16(ct) && al16(stt) && (hd / 2) % 8 == 0) {
    const long long n = (long long)T * nheads * (hd / 16);
    ls::rope_fwd_vec_kernel<<<grid1d(n, 256), 256, 0, st>>>(qkv, ld, pos, ct, stt, T, nheads, hd);
  } else {
    const long long n = (long long)T * nheads * (hd / 2);
    ls::rope_fwd_kernel<<<grid1d(n, 256), 256, 0, st>>>(qkv, ld, pos, ct, stt, T, nheads, hd);
  }
  return cudaGetLastError();
}
cudaError_t rope_bwd_cast(const float* g, bf16* out, long long ld, const int* pos, const float* ct, const float* stt,
                          int T, int nrot, int hd, int ncols, cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  if (ld % 8 == 0 && al16(g) && al16(out) && al16(ct) && al16(stt) && (hd / 2) % 4 == 0 &&
      (ncols - nrot * hd) % 8 == 0 && ncols >= nrot * hd) {
    const long long n = (long long)T * (nrot * (hd / 8) + (ncols - nrot * hd) / 8);
    ls::rope_bwd_cast_vec_kernel<<<grid1d(n, 256), 256, 0, st>>>(g, out, ld, pos, ct, stt, T, nrot, hd, ncols);
  } else {
    const long long n = (long long)T * ncols;
    ls::rope_bwd_cast_kernel<<<grid1d(n, 256), 256, 0, st>>>(g, out, ld, pos, ct, stt, T, nrot, hd, ncols);
  }
  return cudaGetLastError();
}

cudaError_t gemm(int mode, const bf16* A, long long lda, int M, const uint8_t* Wp, const float* Wa, int Nw, int Kw,
                 const bf16* ext_a, const bf16* ext_b, int ext_k, int epi, void* out, long long ldo,
                 const bf16* residual, long long ldr, cudaStream_t st, ls::SkWorkspace sk = {}, int force_bn = 0,
                 int force_nacc = 0, int split = 0) {
  GemmCall c{};
  c.mode = mode;
  c.A = A;
  c.lda = lda;
  c.Wp = Wp;
  c.ext_a = ext_a;
  c.force_bn = force_bn;
  c.force_nacc = force_nacc;
  c.sk = sk;
  c.split = split;
  GemmArgs& g = c.g;
  g.M = M;
  g.Nw = Nw;
  g.Kw = Kw;
  g.Nout = mode == ls::GEMM_FWD ? Nw : Kw;
  g.Kred = mode == ls::GEMM_FWD ? Kw : Nw;
  g.absmax = Wa;
  g.ext_k = ext_k;
  g.ext_b = ext_b;
  g.epi = epi;
  g.out = out;
  g.ldo = ldo;
  g.residual = residual;
  g.ldr = ldr;
  if (M <= 0) return cudaSuccess;
  return ls::launch_nf4_gemm(c, st);
}

// The tensor-core forward: qkv and out 16-byte aligned, ld and ldo multiples of 8.
template <int HD>
cudaError_t attn_fwd_tc_launch(const bf16* qkv, long long ld, const int* cu, int nseq, int maxlen, int nh, int nkv,
                               bf16* out, long long ldo, float* lse, int T, cudaStream_t st) {
  using C = ls::AttnTcCfg<HD>;
  if (T <= 0) return cudaSuccess;
  static std::atomic<uint64_t> attr{0};
  {
    const cudaError_t e = ls::ensure_smem_attr(ls::attn_fwd_tc_kernel<HD>, C::SMEM, attr);
    if (e != cudaSuccess) return e;
  }
  CUtensorMap tm;
  if (!ls::make_map_2d(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, qkv, (uint64_t)ld, (uint64_t)T, (uint64_t)ld * 2, 64,
                       64, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  const int ntq = (maxlen + C::BM - 1) / C::BM;
  dim3 grid((unsigned)nh, (unsigned)nseq, (unsigned)ntq);
  ls::attn_fwd_tc_kernel<HD><<<grid, C::THREADS, C::SMEM, st>>>(tm, cu, nh, nkv, 1.0f / sqrtf((float)HD), out, ldo,
                                                                 lse, T, ntq);
  return cudaGetLastError();
}

// The tensor-core backward: qkv, dout and dqkv 16-byte aligned; ld, lddo multiples of 8,
// ldg of 4.  part (fp32, >= (nh / nkv) * T * 2 * nkv * HD): dK / dV per query head in
// separate CTAs, summed in head order by a second kernel; without it one CTA takes the
// whole key/value group.
template <int HD>
cudaError_t attn_bwd_tc_launch(const bf16* qkv, long long ld, const bf16* dout, const bf16* o, long long lddo,
                               const float* lse, const int* cu, int nseq, int maxlen, int nh, int nkv, float* D,
                               float* dqkv, long long ldg, int T, cudaStream_t st, float* part) {
  using C = ls::AttnBwdTcCfg<HD>;
  if (T <= 0) return cudaSuccess;
  static std::atomic<uint64_t> attr_q{0}, attr_k{0};
  {
    cudaError_t e = ls::ensure_smem_attr(ls::attn_bwd_dq_tc_kernel<HD>, C::SMEM_Q, attr_q);
    if (e == cudaSuccess) e = ls::ensure_smem_attr(ls::attn_bwd_dkdv_tc_kernel<HD>, C::SMEM_K, attr_k);
    if (e != cudaSuccess) return e;
  }
  CUtensorMap tq, td;
  if (!ls::make_map_2d(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, qkv, (uint64_t)ld, (uint64_t)T, (uint64_t)ld * 2, 64,
                       64, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !ls::make_map_2d(&td, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, dout, (uint64_t)lddo, (uint64_t)T, (uint64_t)lddo * 2,
                       64, 64, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  const float scale = 1.0f / sqrtf((float)HD);
  {
    const long long w = (long long)T * nh;
    ls::attn_bwd_dot_kernel<<<(unsigned)((w + 7) / 8), 256, 0, st>>>(dout, o, lddo, nh, HD, D, T);
  }
  const int nt = (maxlen + 127) / 128;
  ls::attn_bwd_dq_tc_kernel<HD><<<dim3((unsigned)nh, (unsigned)nseq, (unsigned)nt), C::THREADS, C::SMEM_Q, st>>>(
      tq, td, lse, D, cu, nh, nkv, scale, dqkv, ldg, T, nt);
  const int hsplit = part ? nh / nkv : 1;
  ls::attn_bwd_dkdv_tc_kernel<HD>
      <<<dim3((unsigned)(nkv * hsplit), (unsigned)nseq, (unsigned)nt), C::THREADS, C::SMEM_K, st>>>(
          tq, td, lse, D, cu, nh, nkv, scale, dqkv, ldg, T, hsplit, part);
  if (hsplit > 1) {
    const long long n4 = (long long)T * 2 * nkv * HD / 4;
    ls::attn_dkdv_reduce_kernel<<<grid1d(n4, 256), 256, 0, st>>>(part, hsplit, nh, nkv, HD, T, dqkv, ldg);
  }
  return cudaGetLastError();
}

cudaError_t attn_fwd(int hd, const bf16* qkv, long long ld, const int* cu, int nseq, int maxlen, int nh, int nkv,
                     bf16* out, long long ldo, float* lse, int T, cudaStream_t st) {
  return hd == 64 ? attn_fwd_tc_launch<64>(qkv, ld, cu, nseq, maxlen, nh, nkv, out, ldo, lse, T, st)
                  : attn_fwd_tc_launch<128>(qkv, ld, cu, nseq, maxlen, nh, nkv, out, ldo, lse, T, st);
}
cudaError_t attn_bwd(int hd, const bf16* qkv, long long ld, const bf16* dout, const bf16* o, long long lddo,
                     const float* lse, const int* cu, int nseq, int maxlen, int nh, int nkv, float* D, float* dqkv,
                     long long ldg, int T, cudaStream_t st, float* part = nullptr) {
  return hd == 64
             ? attn_bwd_tc_launch<64>(qkv, ld, dout, o, lddo, lse, cu, nseq, maxlen, nh, nkv, D, dqkv, ldg, T, st, part)
             : attn_bwd_tc_launch<128>(qkv, ld, dout, o, lddo, lse, cu, nseq, maxlen, nh, nkv, D, dqkv, ldg, T, st,
                                       part);
}

cudaError_t lora_outer(const bf16* X, long long ldx, int ncols, const float* Uf, const bf16* Ub, int ldu, int r, int T,
                       int layout, int accumulate, float* scratch, int rows_per_chunk, float* out, cudaStream_t st) {
  const int nch = (int)(((long long)T + rows_per_chunk - 1) / rows_per_chunk);
  dim3 g1((ncols + 63) / 64, nch);
  ls::lora_outer_partial_kernel<<<g1, 256, 0, st>>>(X, ldx, ncols, Uf, Ub, ldu, r, T, rows_per_chunk, scratch);
  const int n = ncols * r;
  ls::lora_outer_reduce_kernel<<<(n + 255) / 256, 256, 0, st>>>(scratch, nch, ncols, r, layout, accumulate, out);
  return cudaGetLastError();
}

// LoRA projection: with scratch (>= nsplit * T * 32 floats) K is split over
// kLoraSplit blocks per 16-row tile and reduced in slice order by a second kernel
// (more blocks in flight); without it, one block per tile.
constexpr int kLoraSplit = kLoraSplitMax;

cudaError_t lora_proj(const bf16* X, long long ldx, int T, ls::LoraProjHalf h0, ls::LoraProjHalf h1, int r, float s,
                      float* out_f32, bf16* out_ext, float* scratch, cudaStream_t st) {
  const int ns = scratch ? kLoraSplit : 1;
  // 16-byte row reads when every half's columns allow them
  auto v16 = [&](const ls::LoraProjHalf& h) {
    return !h.w || (h.xcol % 8 == 0 && h.K % 32 == 0 &&
                    (h.trans || (h.ldw % 8 == 0 && (reinterpret_cast<uintptr_t>(h.w) & 15) == 0)));
  };
  const dim3 grid((T + 15) / 16, ns);
  if (ldx % 8 == 0 && (reinterpret_cast<uintptr_t>(X) & 15) == 0 && v16(h0) && v16(h1))
    ls::lora_proj_kernel<true><<<grid, 256, 0, st>>>(X, ldx, T, h0, h1, r, s, out_f32, out_ext, scratch);
  else
    ls::lora_proj_kernel<false><<<grid, 256, 0, st>>>(X, ldx, T, h0, h1, r, s, out_f32, out_ext, scratch);
  if (ns > 1)
    ls::lora_proj_reduce_kernel<<<(T * 32 + 255) / 256, 256, 0, st>>>(scratch, ns, T, s, out_f32, out_ext);
  return cudaGetLastError();
}

// LoRA down-projection u_ext = [bf16(s x A_q^T) | bf16(s x A_v^T) | 0].
cudaError_t lora_down(const bf16* x, long long ldx, const bf16* aq, const bf16* av, int r, int K, float s,
                      bf16* u_ext, int T, cudaStream_t st, float* scratch = nullptr) {
  ls::LoraProjHalf h0{aq, (long long)K, 0, K, 0}, h1{av, (long long)K, 0, K, 0};
  return lora_proj(x, ldx, T, h0, h1, r, s, nullptr, u_ext, scratch, st);
}

// du = s [dY_q B_q | dY_v B_v] (fp32 [T, 32]) and its bf16 extra-stage copy du_ext [T, 64].
cudaError_t lora_du(const bf16* dy, long long ldy, int col_q, int nq, const bf16* bq, int col_v, int nv,
                    const bf16* bv, int r, float s, float* du, bf16* du_ext, int T, cudaStream_t st,
                    float* scratch = nullptr) {
  ls::LoraProjHalf h0{bq, 0, col_q, nq, 1}, h1{bv, 0, col_v, nv, 1};
  return lora_proj(dy, ldy, T, h0, h1, r, s, du, du_ext, scratch, st);
}

void CUDART_CB host_sleep(void* p) {
  const int ms = *reinterpret_cast<int*>(p);
  std::this_thread::sleep_for(std::chrono::milliseconds(ms));
}

}  // namespace

// ====================================================================== streaming engine

namespace {

size_t item_layer_component_bytes(const ls_ctx* c, int m, bool absmax) {
  const size_t H = c->H, I = c->I, nq = c->nq, nkv = c->nkvd;
  const size_t rows[7] = {nq, nkv, nkv, H, I, I, H};
  const size_t cols[7] = {H, H, H, nq, H, H, I};
  return absmax ? rows[m] * (cols[m] / 64) * 4 : rows[m] * cols[m] / 2;
}

// Read a file-backed layer image into the next pinned staging buffer (host, now) and
// enqueue its copy into the slot.  The buffer is reused only after its previous copy
// has finished (bounded host wait).  O_DIRECT reads bypass the page cache where the
// file system allows them; the image is read whole (rounded up to 4 KiB).
int copy_item_file(ls_ctx* c, int item, uint8_t* img, cudaStream_t st) {
  if (c->stage.empty()) return fail(c, LS_ERR_STATE, "file-backed layer without staging buffers (ls_set_staging)");
  const int k = c->stage_next;
  c->stage_next = (k + 1) % (int)c->stage.size();
  if (c->stage_used[k]) {
    const auto t0 = std::chrono::steady_clock::now();
    for (;;) {
      const cudaError_t q = cudaEventQuery(c->stage_ev[k]);
      if (q == cudaSuccess) break;
      if (q != cudaErrorNotReady) return fail(c, LS_ERR_CUDA, std::string("staging wait: ") + cudaGetErrorString(q));
      if (std::chrono::steady_clock::now() - t0 > std::chrono::seconds(120))
        return fail(c, LS_ERR_TIMEOUT, "staging buffer still being copied after 120 s");
      std::this_thread::sleep_for(std::chrono::microseconds(50));
    }
  }
  const ls_ctx::FileSrc& f = c->lf[item];
  const size_t n = c->lay.bytes;
  const size_t want = f.direct ? align_up(n, 4096) : n;
  const auto t0 = std::chrono::steady_clock::now();
  size_t got = 0;
  while (got < want) {
    const ssize_t r = pread(f.fd, c->stage[k] + got, want - got, (off_t)(f.off + got));
    if (r < 0) {
      if (errno == EINTR) continue;
      return fail(c, LS_ERR_ARG, std::string("layer file read: ") + strerror(errno));
    }
    if (r == 0) {
      if (got >= n) break;   // the padding past the last image may be missing
      return fail(c, LS_ERR_ARG, "layer file shorter than its image");
    }
    got += (size_t)r;
  }
  c->file_ms += std::chrono::duration<double, std::milli>(std::chrono::steady_clock::now() - t0).count();
  c->file_bytes += n;
  CK(cudaMemcpyAsync(img, c->stage[k], n, cudaMemcpyHostToDevice, st));
  CK(cudaEventRecord(c->stage_ev[k], st));
  c->stage_used[k] = 1;
  c->st.layer_reads++;
  c->st.h2d_bytes += n;
  return LS_OK;
}

int copy_item(ls_ctx* c, int item, uint8_t* img, cudaStream_t st) {
  if (c->copy_delay_ms > 0) CK(cudaLaunchHostFunc(st, host_sleep, &c->copy_delay_ms));
  if (item < c->L && c->lf[item].fd >= 0) return copy_item_file(c, item, img, st);
  if (item < c->L) {
    const ls_layer_host& h = c->hl[item];
    const ls_nf4_host* m7[7] = {&h.q, &h.k, &h.v, &h.o, &h.gate, &h.up, &h.down};
    const void* src[16];
    size_t sz[16];
    for (int m = 0; m < 7; ++m) {
      src[m] = m7[m]->packed;
      sz[m] = item_layer_component_bytes(c, m, false);
      src[7 + m] = m7[m]->absmax;
      sz[7 + m] = item_layer_component_bytes(c, m, true);
    }
    src[14] = h.attn_norm;
    sz[14] = (size_t)c->H * 2;
    src[15] = h.mlp_norm;
    sz[15] = (size_t)c->H * 2;
    // one copy when the host image already has the slot layout
    const uint8_t* hb = reinterpret_cast<const uint8_t*>(src[0]) - c->lay.off[0];
    bool contiguous = true;
    for (int i = 0; i < 16; ++i)
      if (reinterpret_cast<const uint8_t*>(src[i]) != hb + c->lay.off[i]) contiguous = false;
    if (contiguous) {
      CK(cudaMemcpyAsync(img, hb, c->lay.off[15] + sz[15], cudaMemcpyHostToDevice, st));
    } else {
      for (int i = 0; i < 16; ++i) CK(cudaMemcpyAsync(img + c->lay.off[i], src[i], sz[i], cudaMemcpyHostToDevice, st));
    }
    c->st.layer_reads++;
    c->st.h2d_bytes += c->lay.off[15] + sz[15];
  } else {
    const int ch = item - c->L;
    const ls_nf4_host& m = c->cfg.tied ? c->hv.embed : c->hv.lm_head;
    const size_t v0 = (size_t)ch * c->vrows;
    const size_t n = std::min((size_t)c->vrows, (size_t)c->V - v0);
    const size_t pb = n * (c->H / 2), ab = n * (c->H / 64) * 4;
    CK(cudaMemcpyAsync(img, m.packed + v0 * (c->H / 2), pb, cudaMemcpyHostToDevice, st));
    CK(cudaMemcpyAsync(img + c->vch_abs_off, m.absmax + v0 * (c->H / 64), ab, cudaMemcpyHostToDevice, st));
    c->st.vocab_reads++;
    c->st.h2d_bytes += pb + ab;
  }
  return LS_OK;
}

// Start bringing `item` into a slot (unless one already holds it); returns the slot.
int prefetch(ls_ctx* c, int item, int busy, int* slot_out) {
  for (int s = 0; s < 2; ++s)
    if (c->slot_item[s] == item) {
      c->st.slot_reuses++;
      *slot_out = s;
      return LS_OK;
    }
  int v;
  if (busy >= 0) v = 1 - busy;
  else v = c->slot_use[0] <= c->slot_use[1] ? 0 : 1;
  if (c->free_rec[v]) CK(cudaStreamWaitEvent(c->cp, c->ev_free[v], 0));
  c->slot_item[v] = -1;
  int rc = copy_item(c, item, c->slot[v], c->cp);
  if (rc) return rc;
  CK(cudaEventRecord(c->ev_ready[v], c->cp));
  c->slot_item[v] = item;
  *slot_out = v;
  return LS_OK;
}

// Run body(item, image) over items in order, double-buffering the host->device copies.
int run_items(ls_ctx* c, const std::vector<int>& items, const std::function<int(int, uint8_t*)>& body) {
  if (items.empty()) return LS_OK;
  if (c->cfg.resident) {
    for (int it : items) {
      if (!c->res_loaded[it]) {
        int rc = copy_item(c, it, c->res_img[it], c->cs);
        if (rc) return rc;
        c->res_loaded[it] = 1;
      }
      int rc = body(it, c->res_img[it]);
      if (rc) return rc;
    }
    return LS_OK;
  }
  int s_cur;
  int rc = prefetch(c, items[0], -1, &s_cur);
  if (rc) return rc;
  for (size_t j = 0; j < items.size(); ++j) {
    CK(cudaStreamWaitEvent(c->cs, c->ev_ready[s_cur], 0));
    int s_next = -1;
    // A RAM-backed next item is queued on the copy stream first, so the link starts at
    // once.  A file-backed one is read on this host thread (pread): queue this item's
    // kernels first, so the GPU computes while the disk read runs.
    const bool next_file = j + 1 < items.size() && items[j + 1] < c->L && c->lf[items[j + 1]].fd >= 0;
    if (j + 1 < items.size() && !next_file) {
      rc = prefetch(c, items[j + 1], s_cur, &s_next);
      if (rc) return rc;
    }
    c->slot_use[s_cur] = ++c->use_clock;
    rc = body(items[j], c->slot[s_cur]);
    if (rc) return rc;
    if (next_file) {
      rc = prefetch(c, items[j + 1], s_cur, &s_next);
      if (rc) return rc;
    }
    CK(cudaEventRecord(c->ev_free[s_cur], c->cs));
    c->free_rec[s_cur] = true;
    s_cur = s_next;
  }
  return LS_OK;
}

struct LayerW {
  const uint8_t *pqkv, *po, *pgu, *pd;
  const float *aqkv, *ao, *agu, *ad;
  const bf16 *w1, *w2;
};

LayerW layer_ptrs(const ls_ctx* c, uint8_t* img) {
  LayerW w;
  w.pqkv = img + c->lay.off[0];
  w.po = img + c->lay.off[3];
  w.pgu = img + c->lay.off[4];
  w.pd = img + c->lay.off[6];
  w.aqkv = reinterpret_cast<const float*>(img + c->lay.off[7]);
  w.ao = reinterpret_cast<const float*>(img + c->lay.off[10]);
  w.agu = reinterpret_cast<const float*>(img + c->lay.off[11]);
  w.ad = reinterpret_cast<const float*>(img + c->lay.off[13]);
  w.w1 = reinterpret_cast<const bf16*>(img + c->lay.off[14]);
  w.w2 = reinterpret_cast<const bf16*>(img + c->lay.off[15]);
  return w;
}

inline double attn_flop(const ls_ctx* c, int T, int nseq) {
  const double Ls = (double)T / nseq;   // host view: equal sequence lengths
  return 4.0 * c->hd * c->nh * nseq * Ls * (Ls + 1) / 2;
}

// Forward of one decoder layer up to (recompute == true) the MLP input projections,
// or to the layer output x_out.
int layer_forward(ls_ctx* c, const LayerW& w, int layer, const bf16* x_in, bf16* x_out, int T, int nseq,
                  const int32_t* cu, bool adapter, bool recompute, int lora_rows = -1) {
  // rows [0, lora_rows) take the adapter; the extra stage reads zero u rows beyond them
  if (lora_rows < 0) lora_rows = T;
  cudaStream_t st = c->cs;
  const int H = c->H, I = c->I;
  const double TH = (double)T * H;
  GEMM_T(LS_K_OTHER, 0, 4 * TH, rmsnorm_fwd(x_in, w.w1, c->n1, c->rstd1, T, H, c->cfg.eps, st));
  const ls_ctx::Ad& a = c->ad[layer];
  const bool use = adapter && a.on;
  if (use) {
    TIMED(LS_K_OTHER, 2.0 * lora_rows * 2 * c->r * H, 2.0 * lora_rows * H, 2,
          lora_down(c->n1, H, a.aq, a.av, c->r, H, c->cfg.lora_scale, c->u_ext, lora_rows, st, c->lora_part));
    const int n = c->nqkv * 64;
    TIMED(LS_K_OTHER, 0, 2.0 * n, 1,
          ls::build_ext_fwd_kernel<<<(n + 255) / 256, 256, 0, st>>>(a.bq, 0, c->nq, a.bv, c->nq + c->nkvd, c->nkvd,
                                                                    c->r, c->nqkv, c->ext_fwd));
  }
  const int ek = use ? 32 : 0;
  GEMM_T(LS_K_GEMM_FWD, gemm_flop(0, T, c->nqkv, H, ek), gemm_bytes(0, T, c->nqkv, H, 2, false),
         gemm(ls::GEMM_FWD, c->n1, H, T, w.pqkv, w.aqkv, c->nqkv, H, c->u_ext, c->ext_fwd, ek, ls::EPI_BF16, c->qkv,
              c->nqkv, nullptr, 0, st, gemm_ws(c)));
  GEMM_T(LS_K_OTHER, 0, 8.0 * T * (c->nh + c->nkv) * c->hd,
         rope_fwd(c->qkv, c->nqkv, c->pos, c->rope_cos, c->rope_sin, T, c->nh + c->nkv, c->hd, st));
  GEMM_T(LS_K_ATTN_FWD, attn_flop(c, T, nseq), 2.0 * T * (c->nqkv + c->nq),
         attn_fwd(c->hd, c->qkv, c->nqkv, cu, nseq, c->maxlen, c->nh, c->nkv, c->attn_o, c->nq, c->lse_attn, T, st));
  GEMM_T(LS_K_GEMM_FWD, gemm_flop(0, T, H, c->nq, 0), gemm_bytes(0, T, H, c->nq, 2, true),
         gemm(ls::GEMM_FWD, c->attn_o, c->nq, T, w.po, w.ao, H, c->nq, nullptr, nullptr, 0, ls::EPI_BF16, c->x1, H,
              x_in, H, st, gemm_ws(c)));
  GEMM_T(LS_K_OTHER, 0, 4 * TH, rmsnorm_fwd(c->x1, w.w2, c->n2, c->rstd2, T, H, c->cfg.eps, st));
  GEMM_T(LS_K_GEMM_FWD, gemm_flop(0, T, 2 * I, H, 0), gemm_bytes(0, T, 2 * I, H, 2, false),
         gemm(ls::GEMM_FWD, c->n2, H, T, w.pgu, w.agu, 2 * I, H, nullptr, nullptr, 0, ls::EPI_BF16, c->gu, 2 * I,
              nullptr, 0, st, gemm_ws(c)));
  if (recompute) return LS_OK;
  {
    const long long n = (long long)T * (I / 8);
    TIMED(LS_K_OTHER, 0, 6.0 * T * I, 1,
          ls::swiglu_fwd_kernel<<<grid1d(n, 256), 256, 0, st>>>(c->gu, c->hbuf, T, I));
  }
  GEMM_T(LS_K_GEMM_FWD, gemm_flop(0, T, H, I, 0), gemm_bytes(0, T, H, I, 2, true),
         gemm(ls::GEMM_FWD, c->hbuf, I, T, w.pd, w.ad, H, I, nullptr, nullptr, 0, ls::EPI_BF16, x_out, H, c->x1, H,
              st, gemm_ws(c)));
  return LS_OK;
}

// Backward of one layer: gx (fp32, dL/d layer output) becomes dL/d layer input;
// gx_bf mirrors it in bf16.  LoRA gradients are added into the bound buffers.
int layer_backward(ls_ctx* c, const LayerW& w, int layer, const bf16* x_in, int T, int nseq, const int32_t* cu) {
  cudaStream_t st = c->cs;
  const int H = c->H, I = c->I;
  const double TH = (double)T * H;
  const ls_ctx::Ad& a = c->ad[layer];
  int rc = layer_forward(c, w, layer, x_in, nullptr, T, nseq, cu, true, true);
  if (rc) return rc;
  // MLP
  GEMM_T(LS_K_GEMM_DX, gemm_flop(1, T, H, I, 0), gemm_bytes(1, T, H, I, 4, false),
         gemm(ls::GEMM_DX, c->gx_bf, H, T, w.pd, w.ad, H, I, nullptr, nullptr, 0, ls::EPI_F32, c->dh, I, nullptr, 0,
              st, gemm_ws(c)));
  {
    const long long n = (long long)T * (I / 4);
    TIMED(LS_K_OTHER, 0, 12.0 * T * I, 1,
          ls::swiglu_bwd_kernel<<<grid1d(n, 256), 256, 0, st>>>(c->dh, c->gu, c->dgu, T, I));
  }
  GEMM_T(LS_K_GEMM_DX, gemm_flop(1, T, 2 * I, H, 0), gemm_bytes(1, T, 2 * I, H, 4, false),
         gemm(ls::GEMM_DX, c->dgu, 2 * I, T, w.pgu, w.agu, 2 * I, H, nullptr, nullptr, 0, ls::EPI_F32, c->dn, H,
              nullptr, 0, st, gemm_ws(c)));
  GEMM_T(LS_K_OTHER, 0, 16 * TH, rmsnorm_bwd(c->dn, c->x1, c->rstd2, w.w2, c->gx, c->gx_bf, T, H, 1, st));
  // attention
  GEMM_T(LS_K_GEMM_DX, gemm_flop(1, T, H, c->nq, 0), gemm_bytes(1, T, H, c->nq, 2, false),
         gemm(ls::GEMM_DX, c->gx_bf, H, T, w.po, w.ao, H, c->nq, nullptr, nullptr, 0, ls::EPI_BF16, c->do_bf, c->nq,
              nullptr, 0, st, gemm_ws(c)));
  GEMM_T(LS_K_ATTN_BWD, 2 * attn_flop(c, T, nseq), 2.0 * T * (c->nqkv + 2 * c->nq) + 4.0 * T * c->nqkv,
         attn_bwd(c->hd, c->qkv, c->nqkv, c->do_bf, c->attn_o, c->nq, c->lse_attn, cu, nseq, c->maxlen, c->nh,
                  c->nkv, c->Dattn, c->dqkv_f, c->nqkv, T, st, c->nh > c->nkv ? c->attn_part : nullptr));
  c->st.kernel_launches += c->nh > c->nkv ? 3 : 2;
  GEMM_T(LS_K_OTHER, 0, 6.0 * T * c->nqkv,
         rope_bwd_cast(c->dqkv_f, c->dqkv_bf, c->nqkv, c->pos, c->rope_cos, c->rope_sin, T, c->nh + c->nkv, c->hd,
                       c->nqkv, st));
  const bool use = a.on;
  if (use) {
    const float s = c->cfg.lora_scale;
    TIMED(LS_K_OTHER, 2.0 * T * (c->nq + c->nkvd) * c->r, 2.0 * T * (c->nq + c->nkvd), 2,
          lora_du(c->dqkv_bf, c->nqkv, 0, c->nq, a.bq, c->nq + c->nkvd, c->nkvd, a.bv, c->r, s, c->du, c->du_ext,
                  T, st, c->lora_part));
    // dB = dY^T u ;  dA = (s du)^T x
    GEMM_T(LS_K_OTHER, 2.0 * T * c->nq * c->r, 2.0 * T * c->nq,
           lora_outer(c->dqkv_bf, c->nqkv, c->nq, nullptr, c->u_ext, 64, c->r, T, 0, 1, c->lora_part, 128, a.gbq, st));
    GEMM_T(LS_K_OTHER, 2.0 * T * c->nkvd * c->r, 2.0 * T * c->nkvd,
           lora_outer(c->dqkv_bf + c->nq + c->nkvd, c->nqkv, c->nkvd, nullptr, c->u_ext + 16, 64, c->r, T, 0, 1,
                      c->lora_part, 128, a.gbv, st));
    GEMM_T(LS_K_OTHER, 2.0 * TH * c->r, 2 * TH,
           lora_outer(c->n1, H, H, c->du, nullptr, 32, c->r, T, 1, 1, c->lora_part, 128, a.gaq, st));
    GEMM_T(LS_K_OTHER, 2.0 * TH * c->r, 2 * TH,
           lora_outer(c->n1, H, H, c->du + 16, nullptr, 32, c->r, T, 1, 1, c->lora_part, 128, a.gav, st));
    c->st.kernel_launches += 4;
    const int n = H * 64;
    TIMED(LS_K_OTHER, 0, 2.0 * n, 1,
          ls::build_ext_bwd_kernel<<<(n + 255) / 256, 256, 0, st>>>(a.aq, a.av, c->r, H, c->ext_bwd));
  }
  const int ek = use ? 32 : 0;
  GEMM_T(LS_K_GEMM_DX, gemm_flop(1, T, c->nqkv, H, ek), gemm_bytes(1, T, c->nqkv, H, 4, false),
         gemm(ls::GEMM_DX, c->dqkv_bf, c->nqkv, T, w.pqkv, w.aqkv, c->nqkv, H, c->du_ext, c->ext_bwd, ek, ls::EPI_F32,
              c->dn, H, nullptr, 0, st, gemm_ws(c)));
  GEMM_T(LS_K_OTHER, 0, 16 * TH, rmsnorm_bwd(c->dn, x_in, c->rstd1, w.w1, c->gx, c->gx_bf, T, H, 1, st));
  return LS_OK;
}

int sticky(ls_ctx* c) {
  if (!c) return set_thread_err(LS_ERR_ARG, "null context");
  if (c->err) {
    g_thread_err = c->msg;
    return c->err;
  }
  return LS_OK;
}

}  // namespace

// ====================================================================== exported API

extern "C" {

int ls_plan(const ls_config* cfg, uint64_t* device_bytes) {
  std::string why;
  int rc = check_cfg(cfg, why);
  if (rc) return set_thread_err(rc, why);
  Planned p = lay_out(*cfg, nullptr);
  if (device_bytes) *device_bytes = p.total;
  if (cfg->cap_bytes && p.total > cfg->cap_bytes) {
    char b[256];
    snprintf(b, sizeof b, "pre-flight: workspace %.3f GB exceeds the cap %.3f GB", p.total / 1e9,
             cfg->cap_bytes / 1e9);
    return set_thread_err(LS_ERR_CAP, b);
  }
  return LS_OK;
}

int ls_layer_layout(const ls_config* cfg, uint64_t* offsets16, uint64_t* image_bytes) {
  std::string why;
  int rc = check_cfg(cfg, why);
  if (rc) return set_thread_err(rc, why);
  LayerLayout L = layer_layout(*cfg);
  if (offsets16)
    for (int i = 0; i < 16; ++i) offsets16[i] = L.off[i];
  if (image_bytes) *image_bytes = L.bytes;
  return LS_OK;
}

int ls_create(const ls_config* cfg, void* d_workspace, uint64_t ws_bytes, void* compute_stream, void* copy_stream,
              ls_ctx** out) {
  if (!out) return set_thread_err(LS_ERR_ARG, "null output pointer");
  *out = nullptr;
  uint64_t need = 0;
  int rc = ls_plan(cfg, &need);
  if (rc) return rc;
  if (!d_workspace || ws_bytes < need)
    return set_thread_err(LS_ERR_ARG, "workspace missing or smaller than ls_plan's size");
  if (reinterpret_cast<uintptr_t>(d_workspace) % 256) return set_thread_err(LS_ERR_ARG, "workspace not 256-byte aligned");
  if (!compute_stream || !copy_stream || compute_stream == copy_stream)
    return set_thread_err(LS_ERR_ARG, "need two distinct caller streams");
  cudaPointerAttributes pa{};
  if (cudaPointerGetAttributes(&pa, d_workspace) != cudaSuccess || pa.type != cudaMemoryTypeDevice) {
    cudaGetLastError();
    return set_thread_err(LS_ERR_ARG, "workspace is not device memory");
  }
  ls_ctx* c = new ls_ctx();
  c->cfg = *cfg;
  c->cs = reinterpret_cast<cudaStream_t>(compute_stream);
  c->cp = reinterpret_cast<cudaStream_t>(copy_stream);
  c->ws = reinterpret_cast<uint8_t*>(d_workspace);
  c->ws_bytes = ws_bytes;
  c->L = cfg->layers; c->H = cfg->hidden; c->nh = cfg->heads; c->nkv = cfg->kv_heads; c->hd = cfg->head_dim;
  c->I = cfg->inter; c->V = cfg->vocab; c->r = cfg->lora_r;
  c->nq = c->nh * c->hd; c->nkvd = c->nkv * c->hd; c->nqkv = c->nq + 2 * c->nkvd;
  c->Tmax = cfg->max_tokens;
  c->maxlen = cfg->max_seq_len > 0 ? cfg->max_seq_len : cfg->max_tokens;
  c->lay = layer_layout(*cfg);
  Planned p = lay_out(*cfg, c);
  c->hl.assign(c->L, ls_layer_host{});
  c->hl_ok.assign(c->L, 0);
  c->lf.assign(c->L, ls_ctx::FileSrc{});
  c->ad.assign(c->L, ls_ctx::Ad{});
  c->st.workspace_bytes = p.total;
  c->st.slot_bytes = p.slot_bytes;
  c->st.act_store_bytes = p.act_bytes;
  c->st.vocab_chunks = c->nvch;
  c->st.vocab_chunk_rows = c->vrows;
  for (int s = 0; s < 2; ++s) {
    if (cudaEventCreateWithFlags(&c->ev_ready[s], cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&c->ev_free[s], cudaEventDisableTiming) != cudaSuccess) {
      ls_destroy(c);
      return set_thread_err(LS_ERR_CUDA, "event creation failed");
    }
  }
  // RoPE tables
  const int half = c->hd / 2;
  std::vector<float> hc((size_t)c->maxlen * half), hs((size_t)c->maxlen * half);
  ls_rope_table(hc.data(), hs.data(), c->maxlen, c->hd, cfg->rope_theta);
  // the split-tile epoch words start at zero (no launch uses epoch 0)
  if (cudaMemcpyAsync(c->rope_cos, hc.data(), hc.size() * 4, cudaMemcpyHostToDevice, c->cs) != cudaSuccess ||
      cudaMemcpyAsync(c->rope_sin, hs.data(), hs.size() * 4, cudaMemcpyHostToDevice, c->cs) != cudaSuccess ||
      cudaMemsetAsync(c->skw.flags, 0, ls::kSkFlagBytes, c->cs) != cudaSuccess ||
      cudaStreamSynchronize(c->cs) != cudaSuccess) {
    ls_destroy(c);
    return set_thread_err(LS_ERR_CUDA, "rope table upload failed");
  }
  *out = c;
  return LS_OK;
}

int ls_destroy(ls_ctx* c) {
  if (!c) return LS_OK;
  if (c->cs) cudaStreamSynchronize(c->cs);
  if (c->cp) cudaStreamSynchronize(c->cp);
  for (int s = 0; s < 2; ++s) {
    if (c->ev_ready[s]) cudaEventDestroy(c->ev_ready[s]);
    if (c->ev_free[s]) cudaEventDestroy(c->ev_free[s]);
  }
  for (auto& e : c->prof_ev)
    if (e) cudaEventDestroy(e);
  for (auto& e : c->stage_ev)
    if (e) cudaEventDestroy(e);
  for (auto& f : c->files) {
    if (f.second.first >= 0) close(f.second.first);
    if (f.second.second >= 0) close(f.second.second);
  }
  delete c;
  return LS_OK;
}

const char* ls_last_error(const ls_ctx* c) {
  if (c && c->err) return c->msg.c_str();
  return g_thread_err.c_str();
}

int nf4_quantize(const float* w, int64_t rows, int64_t cols, uint8_t* packed, float* absmax, int32_t nthreads) {
  if (!w || !packed || !absmax || rows < 0 || cols <= 0 || cols % 64)
    return set_thread_err(LS_ERR_ARG, "nf4_quantize: null pointer or cols not a positive multiple of 64");
  int nt = nthreads > 0 ? nthreads : (int)std::max(1u, std::thread::hardware_concurrency());
  if (rows < nt * 4) nt = (int)std::max<int64_t>(1, rows / 4);
  std::vector<std::thread> th;
  const int64_t per = (rows + nt - 1) / nt;
  for (int i = 0; i < nt; ++i) {
    const int64_t r0 = i * per, r1 = std::min(rows, r0 + per);
    if (r0 >= r1) break;
    th.emplace_back(quantize_rows, w, r0, r1, cols, packed, absmax);
  }
  for (auto& t : th) t.join();
  return LS_OK;
}

static int check_pinned(const void* p, const char* what, std::string& why) {
  if (!p) { why = std::string(what) + ": null pointer"; return LS_ERR_ARG; }
  cudaPointerAttributes a{};
  cudaError_t e = cudaPointerGetAttributes(&a, p);
  if (e != cudaSuccess || a.type != cudaMemoryTypeHost) {
    cudaGetLastError();
    why = std::string(what) + ": not pinned host memory (use cudaHostAlloc or cudaHostRegister)";
    return LS_ERR_ARG;
  }
  return LS_OK;
}

int load_layer_nf4(ls_ctx* c, int32_t layer, const ls_layer_host* h) {
  int rc = sticky(c);
  if (rc) return rc;
  if (!h || layer < 0 || layer >= c->L) return fail(c, LS_ERR_ARG, "load_layer_nf4: bad layer index or null");
  std::string why;
  const ls_nf4_host* m7[7] = {&h->q, &h->k, &h->v, &h->o, &h->gate, &h->up, &h->down};
  const char* names[7] = {"q", "k", "v", "o", "gate", "up", "down"};
  for (int m = 0; m < 7; ++m) {
    if ((rc = check_pinned(m7[m]->packed, names[m], why)) || (rc = check_pinned(m7[m]->absmax, names[m], why)))
      return set_thread_err(rc, "load_layer_nf4: " + why);
  }
  if ((rc = check_pinned(h->attn_norm, "attn_norm", why)) || (rc = check_pinned(h->mlp_norm, "mlp_norm", why)))
    return set_thread_err(rc, "load_layer_nf4: " + why);
  c->hl[layer] = *h;
  c->hl_ok[layer] = 1;
  c->lf[layer] = ls_ctx::FileSrc{};
  if (c->cfg.resident) c->res_loaded[layer] = 0;
  for (int s = 0; s < 2; ++s)
    if (c->slot_item[s] == layer) c->slot_item[s] = -1;
  return LS_OK;
}

int ls_set_staging(ls_ctx* c, void* h_pinned, uint64_t bytes_each, int32_t nbuf) {
  int rc = sticky(c);
  if (rc) return rc;
  if (!h_pinned || nbuf < 2 || nbuf > 16 || bytes_each < align_up(c->lay.bytes, 4096) || bytes_each % 4096 ||
      reinterpret_cast<uintptr_t>(h_pinned) % 4096)
    return fail(c, LS_ERR_ARG, "ls_set_staging: need 2..16 page-aligned buffers of >= the 4 KiB-rounded layer image");
  std::string why;
  if ((rc = check_pinned(h_pinned, "staging", why))) return set_thread_err(rc, "ls_set_staging: " + why);
  CK(cudaStreamSynchronize(c->cp));
  for (auto& e : c->stage_ev)
    if (e) cudaEventDestroy(e);
  c->stage.clear();
  c->stage_ev.assign(nbuf, nullptr);
  c->stage_used.assign(nbuf, 0);
  for (int i = 0; i < nbuf; ++i) {
    c->stage.push_back(reinterpret_cast<uint8_t*>(h_pinned) + (size_t)i * bytes_each);
    CK(cudaEventCreateWithFlags(&c->stage_ev[i], cudaEventDisableTiming));
  }
  c->stage_bytes = bytes_each;
  c->stage_next = 0;
  return LS_OK;
}

int load_layer_file(ls_ctx* c, int32_t layer, const char* path, uint64_t offset) {
  int rc = sticky(c);
  if (rc) return rc;
  if (!path || layer < 0 || layer >= c->L) return fail(c, LS_ERR_ARG, "load_layer_file: bad layer or null path");
  int fdd = -1, fdb = -1;
  for (auto& f : c->files)
    if (f.first == path) { fdd = f.second.first; fdb = f.second.second; }
  if (fdb < 0) {
    fdb = open(path, O_RDONLY | O_CLOEXEC);
    if (fdb < 0) return set_thread_err(LS_ERR_ARG, std::string("load_layer_file: ") + path + ": " + strerror(errno));
#ifdef O_DIRECT
    fdd = open(path, O_RDONLY | O_CLOEXEC | O_DIRECT);   // -1 where the file system has no direct I/O
#endif
    c->files.push_back({path, {fdd, fdb}});
  }
  const off_t end = lseek(fdb, 0, SEEK_END);
  if (end < 0 || (uint64_t)end < offset + c->lay.bytes)
    return set_thread_err(LS_ERR_ARG, "load_layer_file: file shorter than offset + layer image");
  ls_ctx::FileSrc f;
  f.direct = fdd >= 0 && offset % 4096 == 0;
  f.fd = f.direct ? fdd : fdb;
  f.off = offset;
  c->lf[layer] = f;
  c->hl_ok[layer] = 1;
  if (c->cfg.resident) c->res_loaded[layer] = 0;
  for (int s = 0; s < 2; ++s)
    if (c->slot_item[s] == layer) c->slot_item[s] = -1;
  return LS_OK;
}

int load_vocab_nf4(ls_ctx* c, const ls_vocab_host* h) {
  int rc = sticky(c);
  if (rc) return rc;
  if (!h) return fail(c, LS_ERR_ARG, "load_vocab_nf4: null");
  std::string why;
  if ((rc = check_pinned(h->embed.packed, "embed", why)) || (rc = check_pinned(h->embed.absmax, "embed", why)) ||
      (rc = check_pinned(h->final_norm, "final_norm", why)))
    return set_thread_err(rc, "load_vocab_nf4: " + why);
  if (!c->cfg.tied && ((rc = check_pinned(h->lm_head.packed, "lm_head", why)) ||
                       (rc = check_pinned(h->lm_head.absmax, "lm_head", why))))
    return set_thread_err(rc, "load_vocab_nf4: " + why);
  void* dp = nullptr;
  void* da = nullptr;
  if (cudaHostGetDevicePointer(&dp, const_cast<uint8_t*>(h->embed.packed), 0) != cudaSuccess ||
      cudaHostGetDevicePointer(&da, const_cast<float*>(h->embed.absmax), 0) != cudaSuccess) {
    cudaGetLastError();
    return set_thread_err(LS_ERR_ARG, "load_vocab_nf4: embedding memory is not mapped for device access");
  }
  c->hv = *h;
  c->hv_ok = true;
  c->emb_p = reinterpret_cast<const uint8_t*>(dp);
  c->emb_a = reinterpret_cast<const float*>(da);
  CK(cudaMemcpyAsync(c->wf, h->final_norm, (size_t)c->H * 2, cudaMemcpyHostToDevice, c->cs));
  CK(cudaStreamSynchronize(c->cs));
  for (int i = 0; i < c->nvch; ++i) {
    if (c->cfg.resident) c->res_loaded[c->L + i] = 0;
    for (int s = 0; s < 2; ++s)
      if (c->slot_item[s] == c->L + i) c->slot_item[s] = -1;
  }
  return LS_OK;
}

int ls_set_adapter(ls_ctx* c, int32_t layer, const uint16_t* aq, const uint16_t* bq, const uint16_t* av,
                   const uint16_t* bv, float* gaq, float* gbq, float* gav, float* gbv) {
  int rc = sticky(c);
  if (rc) return rc;
  if (layer < 0 || layer >= c->L) return fail(c, LS_ERR_ARG, "ls_set_adapter: bad layer");
  ls_ctx::Ad a;
  a.aq = reinterpret_cast<const bf16*>(aq); a.bq = reinterpret_cast<const bf16*>(bq);
  a.av = reinterpret_cast<const bf16*>(av); a.bv = reinterpret_cast<const bf16*>(bv);
  a.gaq = gaq; a.gbq = gbq; a.gav = gav; a.gbv = gbv;
  a.on = aq && bq && av && bv;
  if (a.on && !(gaq && gbq && gav && gbv)) return fail(c, LS_ERR_ARG, "ls_set_adapter: gradient buffers missing");
  c->ad[layer] = a;
  return LS_OK;
}

int stream_step_fwd(ls_ctx* c, const int32_t* d_tokens, int32_t T, int32_t nseq, const int32_t* d_cu,
                    const uint8_t* d_mask, int32_t adapter_on, int32_t save_acts, float* d_sums) {
  int rc = sticky(c);
  if (rc) return rc;
  if (!d_tokens || !d_cu || !d_mask || T < 1 || T > c->Tmax || nseq < 1 || nseq > c->cfg.max_seqs)
    return fail(c, LS_ERR_ARG, "stream_step_fwd: bad tokens/offsets/mask or T/nseq outside the configured bounds");
  for (int l = 0; l < c->L; ++l)
    if (!c->hl_ok[l]) return fail(c, LS_ERR_STATE, "stream_step_fwd: layer " + std::to_string(l) + " not loaded");
  if (!c->hv_ok) return fail(c, LS_ERR_STATE, "stream_step_fwd: vocabulary not loaded");
  cudaStream_t st = c->cs;
  const int H = c->H;
  const bool save = save_acts != 0;
  TIMED(LS_K_OTHER, 0, 12.0 * T, 1,
        ls::seq_setup_kernel<<<(T + 255) / 256, 256, 0, st>>>(d_tokens, d_cu, nseq, nullptr, nullptr, c->pos, c->tgt,
                                                             nullptr, T));
  bf16* x0 = save ? c->acts : c->xping;
  {
    const long long n = (long long)T * (H / 8);
    TIMED(LS_K_OTHER, 0, (0.5625 + 2.0) * T * H, 1,
          ls::embed_gather_kernel<<<grid1d(n, 256), 256, 0, st>>>(d_tokens, c->emb_p, c->emb_a, x0, T, H, c->V));
  }
  bf16* hf = save ? c->hf_save : c->hf_tmp;
  float* rstdf = save ? c->rstdf_save : c->rstdf_tmp;
  float* lse = save ? c->lse_save : c->lse_tmp;
  const size_t TH = (size_t)T * H;
  std::vector<int> items;
  for (int l = 0; l < c->L; ++l) items.push_back(l);
  for (int v = 0; v < c->nvch; ++v) items.push_back(c->L + v);
  rc = run_items(c, items, [&](int item, uint8_t* img) -> int {
    if (item < c->L) {
      const int l = item;
      const bf16* xin = save ? c->acts + (size_t)l * (size_t)c->Tmax * H : c->xping + (size_t)(l & 1) * TH;
      bf16* xout = save ? c->acts + (size_t)(l + 1) * (size_t)c->Tmax * H : c->xping + (size_t)((l + 1) & 1) * TH;
      return layer_forward(c, layer_ptrs(c, img), l, xin, xout, T, nseq, d_cu, adapter_on != 0, false);
    }
    const int ch = item - c->L;
    if (ch == 0) {
      const bf16* xL = save ? c->acts + (size_t)c->L * (size_t)c->Tmax * H : c->xping + (size_t)(c->L & 1) * TH;
      GEMM_T(LS_K_OTHER, 0, 4.0 * T * H, rmsnorm_fwd(xL, c->wf, hf, rstdf, T, H, c->cfg.eps, st));
    }
    const int v0 = ch * c->vrows;
    const int n = std::min(c->vrows, c->V - v0);
    GemmCall g{};
    g.mode = ls::GEMM_FWD;
    g.A = hf;
    g.lda = H;
    g.Wp = img;
    g.force_bn = 256;
    g.sk = gemm_ws(c);
    g.g.M = T; g.g.Nw = n; g.g.Kw = H; g.g.Nout = n; g.g.Kred = H;
    g.g.absmax = reinterpret_cast<const float*>(img + c->vch_abs_off);
    g.g.epi = ls::EPI_LOGPROB;
    g.g.targets = c->tgt;
    g.g.vocab_off = v0;
    g.g.part_max = c->pmax; g.g.part_sum = c->psum; g.g.part_ld = c->P;
    g.g.tgt_logit = c->tgt_logit;
    GEMM_T(LS_K_GEMM_FWD, gemm_flop(0, T, n, H, 0), gemm_bytes(0, T, n, H, 0, false) + 8.0 * T * (n / 128),
           ls::launch_nf4_gemm(g, st));
    return LS_OK;
  });
  if (rc) return rc;
  TIMED(LS_K_OTHER, 0, 8.0 * T * c->P, 1,
        ls::logprob_combine_kernel<<<(T + 7) / 8, 256, 0, st>>>(c->pmax, c->psum, c->P, c->P, c->tgt_logit, c->tgt,
                                                               lse, c->lp, T));
  if (d_sums) TIMED(LS_K_OTHER, 0, 5.0 * T, 1, ls::seq_sum_kernel<<<nseq, 256, 0, st>>>(c->lp, d_mask, d_cu, d_sums));
  c->last_T = T;
  c->last_lse = lse;
  if (save) {
    c->saved = true;
    c->s_tokens = d_tokens; c->s_cu = d_cu; c->s_mask = d_mask; c->s_T = T; c->s_nseq = nseq;
  }
  return LS_OK;
}

int stream_step_fwd_dpo(ls_ctx* c, const int32_t* d_tokens, int32_t T, int32_t nseq, const int32_t* d_cu,
                        const uint8_t* d_mask, float* d_pi, float* d_ref) {
  int rc = sticky(c);
  if (rc) return rc;
  if (!c->cfg.dpo_shared_read)
    return fail(c, LS_ERR_STATE, "stream_step_fwd_dpo: context not planned with dpo_shared_read = 1");
  if (!d_tokens || !d_cu || !d_mask || !d_pi || !d_ref || T < 1 || T > c->Tmax || nseq < 1 ||
      nseq > c->cfg.max_seqs)
    return fail(c, LS_ERR_ARG, "stream_step_fwd_dpo: bad buffers or T/nseq outside the configured bounds");
  for (int l = 0; l < c->L; ++l)
    if (!c->hl_ok[l]) return fail(c, LS_ERR_STATE, "stream_step_fwd_dpo: layer " + std::to_string(l) + " not loaded");
  if (!c->hv_ok) return fail(c, LS_ERR_STATE, "stream_step_fwd_dpo: vocabulary not loaded");
  struct PairedRows {
    ls_ctx* c;
    PairedRows(ls_ctx* x, int t) : c(x) { c->pair_rows = t; }
    ~PairedRows() { c->pair_rows = 0; }
  } paired(c, T);
  cudaStream_t st = c->cs;
  const int H = c->H, T2 = 2 * T, n2 = 2 * nseq;
  const size_t TH = (size_t)T * H, T2H = (size_t)T2 * H;
  TIMED(LS_K_OTHER, 0, 12.0 * T2, 1,
        ls::pair_setup_kernel<<<(T2 + 255) / 256, 256, 0, st>>>(d_tokens, d_cu, nseq, T, c->tok2, c->cu2));
  TIMED(LS_K_OTHER, 0, 12.0 * T2, 1,
        ls::seq_setup_kernel<<<(T2 + 255) / 256, 256, 0, st>>>(c->tok2, c->cu2, n2, nullptr, nullptr, c->pos,
                                                              c->tgt, nullptr, T2));
  // the reference rows carry no adapter: their rows of the extra-stage input are zero
  CK(cudaMemsetAsync(c->u_ext + (size_t)T * 64, 0, (size_t)T * 64 * sizeof(bf16), st));
  bf16* x0 = c->xping;
  {
    const long long n = (long long)T * (H / 8);
    TIMED(LS_K_OTHER, 0, (0.5625 + 2.0) * T * H, 1,
          ls::embed_gather_kernel<<<grid1d(n, 256), 256, 0, st>>>(d_tokens, c->emb_p, c->emb_a, x0, T, H, c->V));
  }
  CK(cudaMemcpyAsync(x0 + TH, x0, TH * sizeof(bf16), cudaMemcpyDeviceToDevice, st));
  CK(cudaMemcpyAsync(c->acts, x0, TH * sizeof(bf16), cudaMemcpyDeviceToDevice, st));
  if (c->ref_cap) CK(cudaMemcpyAsync(c->ref_cap, x0 + TH, TH * sizeof(bf16), cudaMemcpyDeviceToDevice, st));
  std::vector<int> items;
  for (int l = 0; l < c->L; ++l) items.push_back(l);
  for (int v = 0; v < c->nvch; ++v) items.push_back(c->L + v);
  rc = run_items(c, items, [&](int item, uint8_t* img) -> int {
    if (item < c->L) {
      const int l = item;
      const bf16* xin = c->xping + (size_t)(l & 1) * T2H;
      bf16* xout = c->xping + (size_t)((l + 1) & 1) * T2H;
      int r2 = layer_forward(c, layer_ptrs(c, img), l, xin, xout, T2, n2, c->cu2, true, false, T);
      if (r2) return r2;
      // the policy rows are the activation store entry of the next layer
      CK(cudaMemcpyAsync(c->acts + (size_t)(l + 1) * (size_t)c->Tmax * H, xout, TH * sizeof(bf16),
                         cudaMemcpyDeviceToDevice, st));
      if (c->ref_cap)
        CK(cudaMemcpyAsync(c->ref_cap + (size_t)(l + 1) * TH, xout + TH, TH * sizeof(bf16), cudaMemcpyDeviceToDevice,
                           st));
      return LS_OK;
    }
    const int ch = item - c->L;
    if (ch == 0) {
      const bf16* xL = c->xping + (size_t)(c->L & 1) * T2H;
      GEMM_T(LS_K_OTHER, 0, 4.0 * T2 * H, rmsnorm_fwd(xL, c->wf, c->hf_tmp, c->rstdf_tmp, T2, H, c->cfg.eps, st));
    }
    const int v0 = ch * c->vrows;
    const int n = std::min(c->vrows, c->V - v0);
    GemmCall g{};
    g.mode = ls::GEMM_FWD;
    g.A = c->hf_tmp;
    g.lda = H;
    g.Wp = img;
    g.force_bn = 256;
    g.sk = gemm_ws(c);
    g.g.M = T2; g.g.Nw = n; g.g.Kw = H; g.g.Nout = n; g.g.Kred = H;
    g.g.absmax = reinterpret_cast<const float*>(img + c->vch_abs_off);
    g.g.epi = ls::EPI_LOGPROB;
    g.g.targets = c->tgt;
    g.g.vocab_off = v0;
    g.g.part_max = c->pmax; g.g.part_sum = c->psum; g.g.part_ld = c->P;
    g.g.tgt_logit = c->tgt_logit;
    GEMM_T(LS_K_GEMM_FWD, gemm_flop(0, T2, n, H, 0), gemm_bytes(0, T2, n, H, 0, false) + 8.0 * T2 * (n / 128),
           ls::launch_nf4_gemm(g, st));
    return LS_OK;
  });
  if (rc) return rc;
  TIMED(LS_K_OTHER, 0, 8.0 * T2 * c->P, 1,
        ls::logprob_combine_kernel<<<(T2 + 7) / 8, 256, 0, st>>>(c->pmax, c->psum, c->P, c->P, c->tgt_logit, c->tgt,
                                                                c->lse_tmp, c->lp, T2));
  TIMED(LS_K_OTHER, 0, 5.0 * T, 1, ls::seq_sum_kernel<<<nseq, 256, 0, st>>>(c->lp, d_mask, d_cu, d_pi));
  TIMED(LS_K_OTHER, 0, 5.0 * T, 1, ls::seq_sum_kernel<<<nseq, 256, 0, st>>>(c->lp + T, d_mask, d_cu, d_ref));
  // what the backward reads of the policy pass
  CK(cudaMemcpyAsync(c->hf_save, c->hf_tmp, TH * sizeof(bf16), cudaMemcpyDeviceToDevice, st));
  CK(cudaMemcpyAsync(c->rstdf_save, c->rstdf_tmp, (size_t)T * 4, cudaMemcpyDeviceToDevice, st));
  CK(cudaMemcpyAsync(c->lse_save, c->lse_tmp, (size_t)T * 4, cudaMemcpyDeviceToDevice, st));
  c->last_T = T2;
  c->last_lse = c->lse_tmp;
  c->saved = true;
  c->s_tokens = d_tokens; c->s_cu = d_cu; c->s_mask = d_mask; c->s_T = T; c->s_nseq = nseq;
  return LS_OK;
}

int seq_logprobs(ls_ctx* c, float* d_lp, float* d_lse) {
  int rc = sticky(c);
  if (rc) return rc;
  if (!c->last_T) return fail(c, LS_ERR_STATE, "seq_logprobs: no forward pass yet");
  if (d_lp) CK(cudaMemcpyAsync(d_lp, c->lp, (size_t)c->last_T * 4, cudaMemcpyDeviceToDevice, c->cs));
  if (d_lse) CK(cudaMemcpyAsync(d_lse, c->last_lse, (size_t)c->last_T * 4, cudaMemcpyDeviceToDevice, c->cs));
  return LS_OK;
}

int dpo_loss(ls_ctx* c, const float* d_pi, const float* d_ref, int32_t npairs, float beta, float* d_loss,
             float* d_coeffs) {
  int rc = sticky(c);
  if (rc) return rc;
  if (!d_pi || !d_ref || npairs < 1) return fail(c, LS_ERR_ARG, "dpo_loss: bad arguments");
  TIMED(LS_K_OTHER, 0, 16.0 * npairs, 1, ls::dpo_loss_kernel<<<1, 32, 0, c->cs>>>(d_pi, d_ref, npairs, beta, d_loss, d_coeffs));
  return LS_OK;
}

}  // extern "C"

namespace ls {
__global__ void sft_loss_kernel(const float* sums, int nseq, float count, float* loss, float* coeffs) {
  if (threadIdx.x != 0) return;
  float s = 0.f;
  for (int i = 0; i < nseq; ++i) s += sums[i];
  if (loss) *loss = -s / count;
  if (coeffs)
    for (int i = 0; i < nseq; ++i) coeffs[i] = -1.f / count;
}
}  // namespace ls

extern "C" {

int sft_loss(ls_ctx* c, const float* d_sums, int32_t nseq, float count, float* d_loss, float* d_coeffs) {
  int rc = sticky(c);
  if (rc) return rc;
  if (!d_sums || nseq < 1 || !(count > 0.f)) return fail(c, LS_ERR_ARG, "sft_loss: bad arguments");
  TIMED(LS_K_OTHER, 0, 8.0 * nseq, 1, ls::sft_loss_kernel<<<1, 32, 0, c->cs>>>(d_sums, nseq, count, d_loss, d_coeffs));
  return LS_OK;
}

int simpo_loss(ls_ctx* c, const float* d_pi, const int32_t* d_cu, const uint8_t* d_mask, int32_t npairs, float beta,
               float gamma, float* d_loss, float* d_coeffs) {
  int rc = sticky(c);
  if (rc) return rc;
  if (!d_pi || !d_cu || !d_mask || npairs < 1) return fail(c, LS_ERR_ARG, "simpo_loss: bad arguments");
  const int n = 2 * npairs;
  TIMED(LS_K_OTHER, 0, 16.0 * n, 1,
        ls::pref_loss_kernel<<<1, 256, n * sizeof(float), c->cs>>>(ls::PREF_SIMPO, d_pi, nullptr, d_cu, d_mask, nullptr,
                                                                   n, beta, gamma, 0.f, d_loss, d_coeffs));
  return LS_OK;
}

int orpo_loss(ls_ctx* c, const float* d_pi, const int32_t* d_cu, const uint8_t* d_mask, int32_t npairs, float lambda,
              float* d_loss, float* d_coeffs) {
  int rc = sticky(c);
  if (rc) return rc;
  if (!d_pi || !d_cu || !d_mask || npairs < 1) return fail(c, LS_ERR_ARG, "orpo_loss: bad arguments");
  const int n = 2 * npairs;
  TIMED(LS_K_OTHER, 0, 16.0 * n, 1,
        ls::pref_loss_kernel<<<1, 256, n * sizeof(float), c->cs>>>(ls::PREF_ORPO, d_pi, nullptr, d_cu, d_mask, nullptr,
                                                                   n, 0.f, lambda, 0.f, d_loss, d_coeffs));
  return LS_OK;
}

int kto_loss(ls_ctx* c, const float* d_pi, const float* d_ref, const uint8_t* d_des, int32_t nseq, float beta,
             float lambda_d, float lambda_u, float* d_loss, float* d_coeffs) {
  int rc = sticky(c);
  if (rc) return rc;
  if (!d_pi || !d_ref || nseq < 1) return fail(c, LS_ERR_ARG, "kto_loss: bad arguments");
  TIMED(LS_K_OTHER, 0, 16.0 * nseq, 1,
        ls::pref_loss_kernel<<<1, 32, 0, c->cs>>>(ls::PREF_KTO, d_pi, d_ref, nullptr, nullptr, d_des, nseq, beta,
                                                  lambda_d, lambda_u, d_loss, d_coeffs));
  return LS_OK;
}

int stream_step_bwd(ls_ctx* c, const float* d_coeffs) {
  int rc = sticky(c);
  if (rc) return rc;
  if (!c->saved) return fail(c, LS_ERR_STATE, "stream_step_bwd: no forward pass with save_acts=1");
  if (!d_coeffs) return fail(c, LS_ERR_ARG, "stream_step_bwd: null coefficients");
  cudaStream_t st = c->cs;
  const int T = c->s_T, nseq = c->s_nseq, H = c->H;
  const int32_t* cu = c->s_cu;
  TIMED(LS_K_OTHER, 0, 17.0 * T, 1,
        ls::seq_setup_kernel<<<(T + 255) / 256, 256, 0, st>>>(c->s_tokens, cu, nseq, c->s_mask, d_coeffs, c->pos,
                                                             c->tgt, c->coef, T));
  std::vector<int> items;
  for (int v = c->nvch - 1; v >= 0; --v) items.push_back(c->L + v);
  for (int l = c->L - 1; l >= 0; --l) items.push_back(l);
  bool first_chunk = true;
  rc = run_items(c, items, [&](int item, uint8_t* img) -> int {
    if (item >= c->L) {
      const int ch = item - c->L;
      const int v0 = ch * c->vrows;
      const int n = std::min(c->vrows, c->V - v0);
      const float* wa = reinterpret_cast<const float*>(img + c->vch_abs_off);
      GemmCall g{};
      g.mode = ls::GEMM_FWD;
      g.A = c->hf_save;
      g.lda = H;
      g.Wp = img;
      g.force_bn = 256;
      g.sk = gemm_ws(c);
      g.g.M = T; g.g.Nw = n; g.g.Kw = H; g.g.Nout = n; g.g.Kred = H;
      g.g.absmax = wa;
      g.g.epi = ls::EPI_DLOGITS;
      g.g.out = c->dlogits; g.g.ldo = n;
      g.g.targets = c->tgt; g.g.vocab_off = v0;
      g.g.lse = c->lse_save; g.g.coef = c->coef;
      GEMM_T(LS_K_GEMM_FWD, gemm_flop(0, T, n, H, 0), gemm_bytes(0, T, n, H, 2, false), ls::launch_nf4_gemm(g, st));
      const int epi = first_chunk ? ls::EPI_F32 : ls::EPI_F32_ACC;
      GEMM_T(LS_K_GEMM_DX, gemm_flop(1, T, n, H, 0), gemm_bytes(1, T, n, H, first_chunk ? 4 : 8, false),
             gemm(ls::GEMM_DX, c->dlogits, n, T, img, wa, n, H, nullptr, nullptr, 0, epi, c->dhf, H, nullptr, 0, st, gemm_ws(c)));
      first_chunk = false;
      if (ch == 0) {
        const bf16* xL = c->acts + (size_t)c->L * (size_t)c->Tmax * H;
        GEMM_T(LS_K_OTHER, 0, 12.0 * T * H,
               rmsnorm_bwd(c->dhf, xL, c->rstdf_save, c->wf, c->gx, c->gx_bf, T, H, 0, st));
      }
      return LS_OK;
    }
    const int l = item;
    const bf16* xin = c->acts + (size_t)l * (size_t)c->Tmax * H;
    return layer_backward(c, layer_ptrs(c, img), l, xin, T, nseq, cu);
  });
  return rc;
}

int lora_grads(ls_ctx* c, float* d_flat, int32_t zero_after) {
  int rc = sticky(c);
  if (rc) return rc;
  size_t off = 0;
  for (int l = 0; l < c->L; ++l) {
    const ls_ctx::Ad& a = c->ad[l];
    if (!a.on) continue;
    float* g4[4] = {a.gaq, a.gbq, a.gav, a.gbv};
    const size_t n4[4] = {(size_t)c->r * c->H, (size_t)c->nq * c->r, (size_t)c->r * c->H, (size_t)c->nkvd * c->r};
    for (int i = 0; i < 4; ++i) {
      if (d_flat) CK(cudaMemcpyAsync(d_flat + off, g4[i], n4[i] * 4, cudaMemcpyDeviceToDevice, c->cs));
      if (zero_after) CK(cudaMemsetAsync(g4[i], 0, n4[i] * 4, c->cs));
      off += n4[i];
    }
  }
  return LS_OK;
}

int lora_params(ls_ctx* c, float* d_flat) {
  int rc = sticky(c);
  if (rc) return rc;
  if (!d_flat) return fail(c, LS_ERR_ARG, "lora_params: null output");
  size_t off = 0;
  for (int l = 0; l < c->L; ++l) {
    const ls_ctx::Ad& a = c->ad[l];
    if (!a.on) continue;
    const bf16* p4[4] = {a.aq, a.bq, a.av, a.bv};
    const size_t n4[4] = {(size_t)c->r * c->H, (size_t)c->nq * c->r, (size_t)c->r * c->H, (size_t)c->nkvd * c->r};
    for (int i = 0; i < 4; ++i) {
      TIMED(LS_K_OTHER, 0, 6.0 * n4[i], 1,
            ls::bf16_to_f32_kernel<<<grid1d((long long)n4[i], 256), 256, 0, c->cs>>>(p4[i], d_flat + off,
                                                                                    (long long)n4[i]));
      off += n4[i];
    }
  }
  return LS_OK;
}

int lora_adamw(ls_ctx* c, float* d_master, float* d_m, float* d_v, int32_t step, float lr, float beta1, float beta2,
               float eps, float wd, int32_t zero_grads) {
  int rc = sticky(c);
  if (rc) return rc;
  if (!d_master || !d_m || !d_v || step < 1) return fail(c, LS_ERR_ARG, "lora_adamw: null state or step < 1");
  const float bc1 = (float)(1.0 - std::pow((double)beta1, step));
  const float bc2 = (float)(1.0 - std::pow((double)beta2, step));
  long long off = 0;
  for (int l = 0; l < c->L; ++l) {
    const ls_ctx::Ad& a = c->ad[l];
    if (!a.on) continue;
    ls::AdamLayer L{};
    float* g4[4] = {a.gaq, a.gbq, a.gav, a.gbv};
    const bf16* p4[4] = {a.aq, a.bq, a.av, a.bv};
    const long long n4[4] = {(long long)c->r * c->H, (long long)c->nq * c->r, (long long)c->r * c->H,
                             (long long)c->nkvd * c->r};
    long long nmax = 0;
    for (int i = 0; i < 4; ++i) {
      L.g[i] = g4[i];
      L.p[i] = const_cast<bf16*>(p4[i]);   // the caller bound these buffers and owns them
      L.off[i] = off;
      L.n[i] = n4[i];
      off += n4[i];
      nmax = std::max(nmax, n4[i]);
    }
    dim3 grid(grid1d(nmax, 256, 148), 4);
    TIMED(LS_K_OTHER, 0, 22.0 * (n4[0] + n4[1] + n4[2] + n4[3]), 1,
          ls::adamw_layer_kernel<<<grid, 256, 0, c->cs>>>(L, d_master, d_m, d_v, lr, beta1, beta2, eps, wd, bc1, bc2,
                                                         zero_grads));
  }
  return LS_OK;
}

int ls_sync(ls_ctx* c, int32_t timeout_ms) {
  if (!c) return set_thread_err(LS_ERR_ARG, "null context");
  cudaEvent_t e[2];
  CK(cudaEventCreateWithFlags(&e[0], cudaEventDisableTiming));
  CK(cudaEventCreateWithFlags(&e[1], cudaEventDisableTiming));
  CK(cudaEventRecord(e[0], c->cs));
  CK(cudaEventRecord(e[1], c->cp));
  const auto t0 = std::chrono::steady_clock::now();
  int result = LS_OK;
  for (int i = 0; i < 2; ++i) {
    for (;;) {
      cudaError_t q = cudaEventQuery(e[i]);
      if (q == cudaSuccess) break;
      if (q != cudaErrorNotReady) {
        result = fail(c, LS_ERR_CUDA, std::string("ls_sync: ") + cudaGetErrorString(q));
        break;
      }
      const double ms = std::chrono::duration<double, std::milli>(std::chrono::steady_clock::now() - t0).count();
      if (timeout_ms > 0 && ms > timeout_ms) {
        result = LS_ERR_TIMEOUT;
        g_thread_err = "ls_sync: streams still busy after " + std::to_string(timeout_ms) + " ms";
        break;
      }
      std::this_thread::sleep_for(std::chrono::microseconds(100));
    }
    if (result) break;
  }
  cudaEventDestroy(e[0]);
  cudaEventDestroy(e[1]);
  if (result) return result;
  int dev = 0;
  CK(cudaMemcpyFromSymbol(&dev, ls::g_device_error, sizeof(int)));
  if (dev) return fail(c, LS_ERR_DEVICE, "a kernel raised device error " + std::to_string(dev));
  return LS_OK;
}

int ls_stats(ls_ctx* c, ls_stats_t* out, int32_t reset) {
  if (!c || !out) return set_thread_err(LS_ERR_ARG, "ls_stats: null argument");
  c->st.file_bytes = c->file_bytes;
  c->st.file_read_ms = c->file_ms;
  *out = c->st;
  if (reset) {
    c->st.layer_reads = c->st.vocab_reads = c->st.h2d_bytes = c->st.slot_reuses = 0;
    c->st.kernel_launches = 0;
    c->file_bytes = 0;
    c->file_ms = 0.0;
  }
  return LS_OK;
}

int ls_profile(ls_ctx* c, int32_t enable) {
  if (!c) return set_thread_err(LS_ERR_ARG, "null context");
  if (enable) {
    if (c->prof_ev.empty()) {
      c->prof_ev.resize(2 * kProfMax);
      for (auto& e : c->prof_ev) CK(cudaEventCreate(&e));
      c->prof_cls.resize(kProfMax);
      c->prof_flop.resize(kProfMax);
      c->prof_bytes.resize(kProfMax);
    }
    c->prof_used = 0;
    c->prof_on = true;
  } else {
    c->prof_on = false;
  }
  return LS_OK;
}

int ls_profile_read(ls_ctx* c, ls_profile_t* out) {
  if (!c || !out) return set_thread_err(LS_ERR_ARG, "ls_profile_read: null argument");
  memset(out, 0, sizeof(*out));
  CK(cudaStreamSynchronize(c->cs));
  for (size_t i = 0; i < c->prof_used; ++i) {
    float ms = 0.f;
    CK(cudaEventElapsedTime(&ms, c->prof_ev[2 * i], c->prof_ev[2 * i + 1]));
    const int k = c->prof_cls[i];
    out->launches[k] += 1;
    out->ms[k] += ms;
    out->flop[k] += c->prof_flop[i];
    out->bytes[k] += c->prof_bytes[i];
  }
  return LS_OK;
}

int ls_read_activation(ls_ctx* c, int32_t layer, uint16_t* d_out) {
  int rc = sticky(c);
  if (rc) return rc;
  if (!c->saved) return fail(c, LS_ERR_STATE, "ls_read_activation: no forward pass with save_acts=1");
  if (!d_out || layer < 0 || layer > c->L) return fail(c, LS_ERR_ARG, "ls_read_activation: bad layer or null output");
  const size_t n = (size_t)c->s_T * c->H;
  CK(cudaMemcpyAsync(d_out, c->acts + (size_t)layer * (size_t)c->Tmax * c->H, n * 2, cudaMemcpyDeviceToDevice, c->cs));
  return LS_OK;
}

int ls_capture_reference(ls_ctx* c, uint16_t* d_buf, uint64_t bytes) {
  int rc = sticky(c);
  if (rc) return rc;
  if (!d_buf) {
    c->ref_cap = nullptr;
    c->ref_cap_bytes = 0;
    return LS_OK;
  }
  if (!c->cfg.dpo_shared_read)
    return fail(c, LS_ERR_STATE, "ls_capture_reference: context not planned with dpo_shared_read = 1");
  const uint64_t need = (uint64_t)(c->L + 1) * (uint64_t)c->Tmax * (uint64_t)c->H * 2;
  if (bytes < need || (reinterpret_cast<uintptr_t>(d_buf) & 15))
    return fail(c, LS_ERR_ARG, "ls_capture_reference: buffer smaller than (L+1) * max_tokens * H bf16, or unaligned");
  c->ref_cap = reinterpret_cast<bf16*>(d_buf);
  c->ref_cap_bytes = bytes;
  return LS_OK;
}

int ls_debug_copy_delay(ls_ctx* c, int32_t ms) {
  if (!c) return set_thread_err(LS_ERR_ARG, "null context");
  c->copy_delay_ms = ms > 0 ? ms : 0;
  return LS_OK;
}

// ====================================================================== kernel-level API

#define KCK(expr)                                                                      \
  do {                                                                                 \
    cudaError_t e_ = (expr);                                                           \
    if (e_ != cudaSuccess) return set_thread_err(LS_ERR_CUDA, cudaGetErrorString(e_)); \
  } while (0)
#define KLAUNCH() KCK(cudaGetLastError())
#define STREAM(s) reinterpret_cast<cudaStream_t>(s)

int lsk_nf4_dequant(const uint8_t* packed, const float* absmax, int64_t rows, int32_t cols, uint16_t* out, void* s) {
  if (!packed || !absmax || !out || rows < 0 || cols <= 0 || cols % 64 || misaligned(packed, 4) || misaligned(out, 16))
    return set_thread_err(LS_ERR_ARG, "lsk_nf4_dequant: bad args");
  const long long n = rows * (cols / 8);
  if (n == 0) return LS_OK;
  ls::nf4_dequant_kernel<<<grid1d(n, 256), 256, 0, STREAM(s)>>>(packed, absmax, reinterpret_cast<bf16*>(out), rows, cols);
  KLAUNCH();
  return LS_OK;
}

int lsk_nf4_gemm(int32_t mode, const uint16_t* A, int64_t lda, int32_t M, const uint8_t* wp, const float* wa,
                 int32_t N, int32_t K, const uint16_t* ext_a, const uint16_t* ext_b, int32_t ext_k, int32_t epi,
                 void* out, int64_t ldo, const uint16_t* residual, int64_t ldr, int32_t force_bn, int32_t force_nacc,
                 void* s) {
  if (mode != 0 && mode != 1) return set_thread_err(LS_ERR_ARG, "lsk_nf4_gemm: mode must be 0 or 1");
  if (!A || !wp || !wa || !out || M < 0 || N <= 0 || K <= 0 || K % 64 || N % 64)
    return set_thread_err(LS_ERR_ARG, "lsk_nf4_gemm: null pointer or N, K not positive multiples of 64");
  if (epi < 0 || epi > 2) return set_thread_err(LS_ERR_ARG, "lsk_nf4_gemm: epi must be 0, 1 or 2");
  if (ext_k != 0 && ext_k != 16 && ext_k != 32) return set_thread_err(LS_ERR_ARG, "lsk_nf4_gemm: ext_k must be 0, 16, 32");
  if (ext_k && (!ext_a || !ext_b)) return set_thread_err(LS_ERR_ARG, "lsk_nf4_gemm: ext operands missing");
  const int outc = mode == 0 ? N : K;
  const int red = mode == 0 ? K : N;
  if (lda < red || lda % 8 || ldo < outc || ldo % 8 || (residual && (ldr < outc || ldr % 8)))
    return set_thread_err(LS_ERR_ARG, "lsk_nf4_gemm: leading dimensions too small or not multiples of 8");
  if (force_bn != 0 && force_bn != 128 && force_bn != 256) return set_thread_err(LS_ERR_ARG, "lsk_nf4_gemm: force_bn");
  if (force_nacc < 0 || force_nacc > 2) return set_thread_err(LS_ERR_ARG, "lsk_nf4_gemm: force_nacc");
  if (residual && epi != 0) return set_thread_err(LS_ERR_ARG, "lsk_nf4_gemm: residual only with bf16 output");
  if (misaligned(A, 16) || misaligned(wp, 16) || misaligned(wa, 4) || misaligned(out, 16) || misaligned(residual, 16) ||
      misaligned(ext_a, 16) || misaligned(ext_b, 16))
    return set_thread_err(LS_ERR_ARG, "lsk_nf4_gemm: A, w_packed, ext_a, ext_b, out, residual must be 16-byte aligned, "
                                      "absmax 4-byte");
  KCK(gemm(mode, reinterpret_cast<const bf16*>(A), lda, M, wp, wa, N, K, reinterpret_cast<const bf16*>(ext_a),
           reinterpret_cast<const bf16*>(ext_b), ext_k, epi, out, ldo, reinterpret_cast<const bf16*>(residual), ldr,
           STREAM(s), ls::SkWorkspace{}, force_bn, force_nacc));
  return LS_OK;
}

uint64_t lsk_nf4_gemm_workspace_bytes(void) { return ls::kSkWorkspaceBytes; }

static ls::SkWorkspace paired_ws(void* workspace, int pair_rows) {
  ls::SkWorkspace w = ls::sk_workspace_at(workspace);
  w.pair_rows = pair_rows;
  return w;
}

int lsk_nf4_gemm_plan(int32_t mode, int32_t M, int32_t N, int32_t K, int32_t ext_k, int32_t split,
                      int32_t pair_rows, int32_t with_workspace, int32_t force_bn, int32_t force_nacc, int32_t sms,
                      lsk_gemm_plan* out) {
  if (!out || (mode != 0 && mode != 1) || M < 1 || N <= 0 || K <= 0 || K % 64 || N % 64 ||
      (ext_k != 0 && ext_k != 16 && ext_k != 32) || split < -1 || split > 1 || pair_rows < 0 ||
      (force_bn != 0 && force_bn != 128 && force_bn != 256) || force_nacc < 0 || force_nacc > 2 || sms < 0)
    return set_thread_err(LS_ERR_ARG, "lsk_nf4_gemm_plan: bad args");
  const int g = sms == 0 ? ls::sk_max_ctas() : std::min(sms, ls::kSkMaxCtas);
  const int outc = mode == 0 ? N : K, red = mode == 0 ? K : N;
  ls::GemmPlan p;
  ls::plan_tile(mode, M, outc, red, ext_k, with_workspace != 0, split, force_bn, force_nacc, g, p);
  ls::plan_schedule(M, outc, red, ext_k, g, pair_rows, p);
  out->nacc = p.nacc;
  out->bn = p.bn;
  out->tiles_m = p.tiles_m;
  out->tiles_n = p.tiles_n;
  out->ctas = p.ctas;
  out->whole_per_cta = p.whole_per_cta;
  out->split_iters = p.split_iters;
  out->k_iters = red / 64 + (ext_k > 0 ? 1 : 0);
  out->pair_rows = p.pair_rows;
  return LS_OK;
}

int lsk_nf4_gemm_sk(int32_t mode, const uint16_t* A, int64_t lda, int32_t M, const uint8_t* wp, const float* wa,
                    int32_t N, int32_t K, const uint16_t* ext_a, const uint16_t* ext_b, int32_t ext_k, int32_t epi,
                    void* out, int64_t ldo, const uint16_t* residual, int64_t ldr, int32_t force_bn,
                    int32_t force_nacc, int32_t split, int32_t pair_rows, void* workspace, uint64_t workspace_bytes,
                    void* s) {
  if (split < -1 || split > 1) return set_thread_err(LS_ERR_ARG, "lsk_nf4_gemm_sk: split must be -1, 0 or 1");
  if (pair_rows < 0) return set_thread_err(LS_ERR_ARG, "lsk_nf4_gemm_sk: pair_rows must be >= 0");
  if (!workspace || workspace_bytes < ls::kSkWorkspaceBytes || reinterpret_cast<uintptr_t>(workspace) % 256)
    return set_thread_err(LS_ERR_ARG, "lsk_nf4_gemm_sk: workspace missing, smaller than "
                                      "lsk_nf4_gemm_workspace_bytes() or not 256-byte aligned");
  if (mode != 0 && mode != 1) return set_thread_err(LS_ERR_ARG, "lsk_nf4_gemm_sk: mode must be 0 or 1");
  if (!A || !wp || !wa || !out || M < 0 || N <= 0 || K <= 0 || K % 64 || N % 64)
    return set_thread_err(LS_ERR_ARG, "lsk_nf4_gemm_sk: null pointer or N, K not positive multiples of 64");
  if (epi < 0 || epi > 2) return set_thread_err(LS_ERR_ARG, "lsk_nf4_gemm_sk: epi must be 0, 1 or 2");
  if (ext_k != 0 && ext_k != 16 && ext_k != 32)
    return set_thread_err(LS_ERR_ARG, "lsk_nf4_gemm_sk: ext_k must be 0, 16, 32");
  if (ext_k && (!ext_a || !ext_b)) return set_thread_err(LS_ERR_ARG, "lsk_nf4_gemm_sk: ext operands missing");
  const int outc = mode == 0 ? N : K;
  const int red = mode == 0 ? K : N;
  if (lda < red || lda % 8 || ldo < outc || ldo % 8 || (residual && (ldr < outc || ldr % 8)))
    return set_thread_err(LS_ERR_ARG, "lsk_nf4_gemm_sk: leading dimensions too small or not multiples of 8");
  if (force_bn != 0 && force_bn != 128 && force_bn != 256)
    return set_thread_err(LS_ERR_ARG, "lsk_nf4_gemm_sk: force_bn");
  if (force_nacc < 0 || force_nacc > 2) return set_thread_err(LS_ERR_ARG, "lsk_nf4_gemm_sk: force_nacc");
  if (residual && epi != 0) return set_thread_err(LS_ERR_ARG, "lsk_nf4_gemm_sk: residual only with bf16 output");
  if (misaligned(A, 16) || misaligned(wp, 16) || misaligned(wa, 4) || misaligned(out, 16) || misaligned(residual, 16) ||
      misaligned(ext_a, 16) || misaligned(ext_b, 16))
    return set_thread_err(LS_ERR_ARG, "lsk_nf4_gemm_sk: A, w_packed, ext_a, ext_b, out, residual must be 16-byte aligned, "
                                      "absmax 4-byte");
  KCK(gemm(mode, reinterpret_cast<const bf16*>(A), lda, M, wp, wa, N, K, reinterpret_cast<const bf16*>(ext_a),
           reinterpret_cast<const bf16*>(ext_b), ext_k, epi, out, ldo, reinterpret_cast<const bf16*>(residual), ldr,
           STREAM(s), paired_ws(workspace, pair_rows), force_bn, force_nacc, split));
  return LS_OK;
}

int lsk_rmsnorm_fwd(const uint16_t* x, const uint16_t* w, uint16_t* y, float* rstd, int32_t T, int32_t H, float eps,
                    void* s) {
  if (!x || !w || !y || T < 0 || H <= 0 || H % 8 || misaligned(x, 16) || misaligned(w, 16) || misaligned(y, 16))
    return set_thread_err(LS_ERR_ARG, "lsk_rmsnorm_fwd: bad args");
  if (T == 0) return LS_OK;
  KCK(rmsnorm_fwd(reinterpret_cast<const bf16*>(x), reinterpret_cast<const bf16*>(w), reinterpret_cast<bf16*>(y),
                  rstd, T, H, eps, STREAM(s)));
  return LS_OK;
}

int lsk_rmsnorm_bwd(const float* dy, const uint16_t* x, const float* rstd, const uint16_t* w, float* dx,
                    uint16_t* dx_bf16, int32_t T, int32_t H, int32_t accumulate, void* s) {
  if (!dy || !x || !rstd || !w || !dx || T < 0 || H <= 0 || H % 4 || misaligned(dy, 16) || misaligned(dx, 16) ||
      misaligned(x, 8) || misaligned(w, 8) || misaligned(dx_bf16, 8))
    return set_thread_err(LS_ERR_ARG, "lsk_rmsnorm_bwd: bad args");
  if (T == 0) return LS_OK;
  KCK(rmsnorm_bwd(dy, reinterpret_cast<const bf16*>(x), rstd, reinterpret_cast<const bf16*>(w), dx,
                  reinterpret_cast<bf16*>(dx_bf16), T, H, accumulate, STREAM(s)));
  return LS_OK;
}

int ls_rope_table(float* hc, float* hs, int32_t max_pos, int32_t hd, float theta) {
  if (!hc || !hs || max_pos < 1 || hd < 2 || hd % 2) return set_thread_err(LS_ERR_ARG, "ls_rope_table: bad args");
  const int half = hd / 2;
  for (int i = 0; i < half; ++i) {
    const double inv = std::pow((double)theta, -2.0 * i / hd);
    for (int p = 0; p < max_pos; ++p) {
      const double a = p * inv;
      hc[(size_t)p * half + i] = (float)std::cos(a);
      hs[(size_t)p * half + i] = (float)std::sin(a);
    }
  }
  return LS_OK;
}

int lsk_rope_fwd(uint16_t* qkv, int64_t ld, const int32_t* pos, const float* ct, const float* stt, int32_t T,
                 int32_t nheads, int32_t hd, void* s) {
  if (!qkv || !pos || !ct || !stt || T < 0 || nheads < 1 || hd % 2 || ld < (int64_t)nheads * hd)
    return set_thread_err(LS_ERR_ARG, "lsk_rope_fwd: bad args");
  if ((long long)T * nheads * (hd / 2) == 0) return LS_OK;
  KCK(rope_fwd(reinterpret_cast<bf16*>(qkv), ld, pos, ct, stt, T, nheads, hd, STREAM(s)));
  return LS_OK;
}

int lsk_rope_bwd_cast(const float* g, uint16_t* out, int64_t ld, const int32_t* pos, const float* ct,
                      const float* stt, int32_t T, int32_t nrot, int32_t hd, int32_t ncols, void* s) {
  if (!g || !out || !pos || !ct || !stt || T < 0 || ncols > ld || nrot * hd > ncols)
    return set_thread_err(LS_ERR_ARG, "lsk_rope_bwd_cast: bad args");
  if ((long long)T * ncols == 0) return LS_OK;
  KCK(rope_bwd_cast(g, reinterpret_cast<bf16*>(out), ld, pos, ct, stt, T, nrot, hd, ncols, STREAM(s)));
  return LS_OK;
}

int lsk_attn_fwd(const uint16_t* qkv, int64_t ld, const int32_t* cu, int32_t nseq, int32_t max_len, int32_t nh,
                 int32_t nkv, int32_t hd, uint16_t* out, int64_t ldo, float* lse, int32_t T, void* s) {
  // grid: (query heads, sequences, 128-row query tiles); the last two are limited to 65535
  if (!qkv || !cu || !out || !lse || nseq < 1 || nseq > 65535 || max_len < 1 || (max_len + 127) / 128 > 65535 ||
      nh < 1 || nkv < 1 || nh % nkv || (hd != 64 && hd != 128) || ld < (int64_t)(nh + 2 * nkv) * hd || ld % 8 ||
      ldo < (int64_t)nh * hd || ldo % 8 || (reinterpret_cast<uintptr_t>(qkv) & 15) ||
      (reinterpret_cast<uintptr_t>(out) & 15))
    return set_thread_err(LS_ERR_ARG, "lsk_attn_fwd: bad args");
  KCK(attn_fwd(hd, reinterpret_cast<const bf16*>(qkv), ld, cu, nseq, max_len, nh, nkv, reinterpret_cast<bf16*>(out),
               ldo, lse, T, STREAM(s)));
  return LS_OK;
}

int lsk_attn_bwd(const uint16_t* qkv, int64_t ld, const uint16_t* dout, const uint16_t* o, int64_t lddo,
                 const float* lse, const int32_t* cu, int32_t nseq, int32_t max_len, int32_t nh, int32_t nkv,
                 int32_t hd, float* D, float* dqkv, int64_t ldg, int32_t T, float* part, void* s) {
  const int64_t w = (int64_t)(nh + 2 * nkv) * hd;   // q | k | v columns
  if (!qkv || !dout || !o || !lse || !cu || !D || !dqkv || nseq < 1 || nseq > 65535 || max_len < 1 ||
      (max_len + 127) / 128 > 65535 || nh < 1 || nkv < 1 || nh % nkv || (hd != 64 && hd != 128) || ld < w ||
      ld % 8 || lddo < (int64_t)nh * hd || lddo % 8 || ldg < w || ldg % 4 ||
      ((reinterpret_cast<uintptr_t>(qkv) | reinterpret_cast<uintptr_t>(dout) | reinterpret_cast<uintptr_t>(o) |
        reinterpret_cast<uintptr_t>(dqkv) | reinterpret_cast<uintptr_t>(part)) & 15))
    return set_thread_err(LS_ERR_ARG, "lsk_attn_bwd: bad args");
  KCK(attn_bwd(hd, reinterpret_cast<const bf16*>(qkv), ld, reinterpret_cast<const bf16*>(dout),
               reinterpret_cast<const bf16*>(o), lddo, lse, cu, nseq, max_len, nh, nkv, D, dqkv, ldg, T, STREAM(s),
               nh > nkv ? part : nullptr));
  return LS_OK;
}

int lsk_swiglu_fwd(const uint16_t* gu, uint16_t* h, int32_t T, int32_t I, void* s) {
  if (!gu || !h || T < 0 || I <= 0 || I % 8 || misaligned(gu, 16) || misaligned(h, 16))
    return set_thread_err(LS_ERR_ARG, "lsk_swiglu_fwd: bad args");
  const long long n = (long long)T * (I / 8);
  if (n == 0) return LS_OK;
  ls::swiglu_fwd_kernel<<<grid1d(n, 256), 256, 0, STREAM(s)>>>(reinterpret_cast<const bf16*>(gu), reinterpret_cast<bf16*>(h), T, I);
  KLAUNCH();
  return LS_OK;
}

int lsk_swiglu_bwd(const float* dh, const uint16_t* gu, uint16_t* dgu, int32_t T, int32_t I, void* s) {
  if (!dh || !gu || !dgu || T < 0 || I <= 0 || I % 4 || misaligned(dh, 16) || misaligned(gu, 8) || misaligned(dgu, 8))
    return set_thread_err(LS_ERR_ARG, "lsk_swiglu_bwd: bad args");
  const long long n = (long long)T * (I / 4);
  if (n == 0) return LS_OK;
  ls::swiglu_bwd_kernel<<<grid1d(n, 256), 256, 0, STREAM(s)>>>(dh, reinterpret_cast<const bf16*>(gu), reinterpret_cast<bf16*>(dgu), T, I);
  KLAUNCH();
  return LS_OK;
}

int lsk_lora_down(const uint16_t* x, int64_t ldx, const uint16_t* aq, const uint16_t* av, int32_t r, int32_t K,
                  float sc, uint16_t* u_ext, int32_t T, void* s) {
  if (!x || !u_ext || r < 1 || r > 16 || K <= 0 || K % 8 || ldx < K || ldx % 8 || T < 0 || misaligned(x, 4) ||
      misaligned(aq, 4) || misaligned(av, 4))
    return set_thread_err(LS_ERR_ARG, "lsk_lora_down: bad args");
  if (K % 16) return set_thread_err(LS_ERR_ARG, "lsk_lora_down: K must be a multiple of 16");
  if (T == 0) return LS_OK;
  KCK(lora_down(reinterpret_cast<const bf16*>(x), ldx, reinterpret_cast<const bf16*>(aq),
                reinterpret_cast<const bf16*>(av), r, K, sc, reinterpret_cast<bf16*>(u_ext), T, STREAM(s)));
  return LS_OK;
}

int lsk_lora_du(const uint16_t* dy, int64_t ldy, int32_t col_q, int32_t nq, const uint16_t* bq, int32_t col_v,
                int32_t nv, const uint16_t* bv, int32_t r, float sc, float* du, uint16_t* du_ext, int32_t T, void* s) {
  if (!dy || !du || !du_ext || r < 1 || r > 16 || T < 0 || ldy % 2 || col_q % 2 || col_v % 2 || misaligned(dy, 4) ||
      (bq && (nq < 16 || nq % 16)) || (bv && (nv < 16 || nv % 16)))
    return set_thread_err(LS_ERR_ARG, "lsk_lora_du: bad args (even pitch/offsets, widths multiples of 16)");
  if (T == 0) return LS_OK;
  KCK(lora_du(reinterpret_cast<const bf16*>(dy), ldy, col_q, nq, reinterpret_cast<const bf16*>(bq), col_v, nv,
              reinterpret_cast<const bf16*>(bv), r, sc, du, reinterpret_cast<bf16*>(du_ext), T, STREAM(s)));
  return LS_OK;
}

int lsk_lora_outer(const uint16_t* X, int64_t ldx, int32_t ncols, const float* uf, const uint16_t* ub, int32_t ldu,
                   int32_t r, int32_t T, int32_t layout, int32_t accumulate, float* scratch, int32_t rpc, float* out,
                   void* s) {
  if (!X || (!uf && !ub) || !scratch || !out || r < 1 || r > 16 || ncols < 1 || ncols % 8 || ldx % 8 ||
      ldx < ncols || ldu < r || (reinterpret_cast<uintptr_t>(X) & 15) || misaligned(scratch, 8) || T < 1 || rpc < 1 ||
      (layout != 0 && layout != 1) || ((long long)T + rpc - 1) / rpc > 65535)
    return set_thread_err(LS_ERR_ARG, "lsk_lora_outer: bad args");
  KCK(lora_outer(reinterpret_cast<const bf16*>(X), ldx, ncols, uf, reinterpret_cast<const bf16*>(ub), ldu, r, T,
                 layout, accumulate, scratch, rpc, out, STREAM(s)));
  return LS_OK;
}

}  // extern "C"

// Partial sums of lsk_lora_outer_noalloc: a fixed array in the library image (no
// allocation at run time).  Host code must not use the symbol as an address: its
// device address comes from cudaGetSymbolAddress, looked up once per device.
static __device__ __align__(256) float g_outer_noalloc_scratch[LS_OUTER_NOALLOC_SCRATCH_FLOATS];

namespace {
std::mutex g_noalloc_mu;
constexpr int kMaxDevices = 256;
float* g_noalloc_addr[kMaxDevices] = {};
}  // namespace

extern "C" {

int lsk_lora_outer_noalloc(const uint16_t* X, int64_t ldx, int32_t ncols, const float* uf, const uint16_t* ub,
                           int32_t ldu, int32_t r, int32_t T, int32_t layout, int32_t accumulate, int32_t rpc,
                           float* out, void* s) {
  if (!X || (!uf && !ub) || !out || r < 1 || r > 16 || ncols < 1 || ncols % 8 || ldx % 8 || ldx < ncols ||
      ldu < r || (reinterpret_cast<uintptr_t>(X) & 15) || T < 1 || rpc < 1 || (layout != 0 && layout != 1) ||
      ((long long)T + rpc - 1) / rpc > 65535)
    return set_thread_err(LS_ERR_ARG, "lsk_lora_outer_noalloc: bad args");
  const long long need = (((long long)T + rpc - 1) / rpc) * (long long)ncols * 16;
  if (need > (long long)LS_OUTER_NOALLOC_SCRATCH_FLOATS) {
    char b[200];
    snprintf(b, sizeof b, "lsk_lora_outer_noalloc: needs %lld scratch floats (ceil(T/rows_per_chunk)*ncols*16), "
             "more than the fixed %d", need, (int)LS_OUTER_NOALLOC_SCRATCH_FLOATS);
    return set_thread_err(LS_ERR_ARG, b);
  }
  int dev = -1;
  KCK(cudaGetDevice(&dev));
  if (dev < 0 || dev >= kMaxDevices) return set_thread_err(LS_ERR_ARG, "lsk_lora_outer_noalloc: device ordinal out of range");
  float* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_addr[dev]) {
      void* p = nullptr;
      const cudaError_t e = cudaGetSymbolAddress(&p, g_outer_noalloc_scratch);
      if (e != cudaSuccess || !p)
        return set_thread_err(LS_ERR_CUDA, std::string("lsk_lora_outer_noalloc: cudaGetSymbolAddress: ") +
                                               cudaGetErrorString(e));
      g_noalloc_addr[dev] = reinterpret_cast<float*>(p);
    }
    scratch = g_noalloc_addr[dev];
  }
  KCK(lora_outer(reinterpret_cast<const bf16*>(X), ldx, ncols, uf, reinterpret_cast<const bf16*>(ub), ldu, r, T,
                 layout, accumulate, scratch, rpc, out, STREAM(s)));
  return LS_OK;
}

int lsk_build_ext_fwd(const uint16_t* bq, int32_t q0, int32_t nq, const uint16_t* bv, int32_t v0, int32_t nv,
                      int32_t r, int32_t N, uint16_t* ext, void* s) {
  if (!ext || N < 1 || N > INT_MAX / 64 || r < 1 || r > 16) return set_thread_err(LS_ERR_ARG, "lsk_build_ext_fwd: bad args");
  const int n = N * 64;
  ls::build_ext_fwd_kernel<<<(n + 255) / 256, 256, 0, STREAM(s)>>>(reinterpret_cast<const bf16*>(bq), q0, nq,
                                                                  reinterpret_cast<const bf16*>(bv), v0, nv, r, N,
                                                                  reinterpret_cast<bf16*>(ext));
  KLAUNCH();
  return LS_OK;
}

int lsk_build_ext_bwd(const uint16_t* aq, const uint16_t* av, int32_t r, int32_t K, uint16_t* ext, void* s) {
  if (!ext || K < 1 || K > INT_MAX / 64 || r < 1 || r > 16) return set_thread_err(LS_ERR_ARG, "lsk_build_ext_bwd: bad args");
  const int n = K * 64;
  ls::build_ext_bwd_kernel<<<(n + 255) / 256, 256, 0, STREAM(s)>>>(reinterpret_cast<const bf16*>(aq),
                                                                  reinterpret_cast<const bf16*>(av), r, K,
                                                                  reinterpret_cast<bf16*>(ext));
  KLAUNCH();
  return LS_OK;
}

int lsk_embed_gather(const int32_t* tokens, const uint8_t* packed, const float* absmax, int32_t V, uint16_t* x,
                     int32_t T, int32_t H, void* s) {
  if (!tokens || !packed || !absmax || !x || V < 1 || T < 0 || H % 64 || misaligned(packed, 4) || misaligned(x, 16))
    return set_thread_err(LS_ERR_ARG, "lsk_embed_gather: bad args");
  const long long n = (long long)T * (H / 8);
  if (n == 0) return LS_OK;
  ls::embed_gather_kernel<<<grid1d(n, 256), 256, 0, STREAM(s)>>>(tokens, packed, absmax, reinterpret_cast<bf16*>(x), T,
                                                                 H, V);
  KLAUNCH();
  return LS_OK;
}

int lsk_vocab_logprob(const uint16_t* h, int32_t T, int32_t H, const uint8_t* wp, const float* wa, int32_t V,
                      const int32_t* targets, float* scratch, float* tgt_logit, float* lse, float* lp, void* s) {
  if (!h || !wp || !wa || !targets || !scratch || !tgt_logit || !lse || !lp || T < 1 || H % 64 || V % 64 || V < 64 ||
      misaligned(h, 16) || misaligned(wp, 16) || misaligned(wa, 4))
    return set_thread_err(LS_ERR_ARG, "lsk_vocab_logprob: bad args");
  const int P = (V + 127) / 128;
  float* pmax = scratch;
  float* psum = scratch + (size_t)T * P;
  GemmCall g{};
  g.mode = ls::GEMM_FWD;
  g.A = reinterpret_cast<const bf16*>(h);
  g.lda = H;
  g.Wp = wp;
  g.force_bn = 256;
  g.g.M = T; g.g.Nw = V; g.g.Kw = H; g.g.Nout = V; g.g.Kred = H;
  g.g.absmax = wa;
  g.g.epi = ls::EPI_LOGPROB;
  g.g.targets = targets; g.g.vocab_off = 0;
  g.g.part_max = pmax; g.g.part_sum = psum; g.g.part_ld = P;
  g.g.tgt_logit = tgt_logit;
  KCK(ls::launch_nf4_gemm(g, STREAM(s)));
  ls::logprob_combine_kernel<<<(T + 7) / 8, 256, 0, STREAM(s)>>>(pmax, psum, P, P, tgt_logit, targets, lse, lp, T);
  KLAUNCH();
  return LS_OK;
}

int lsk_vocab_bwd(const uint16_t* h, int32_t T, int32_t H, const uint8_t* wp, const float* wa, int32_t v0, int32_t n,
                  const int32_t* targets, const float* lse, const float* coef, uint16_t* dlogits, float* dh,
                  int32_t accumulate, void* s) {
  if (!h || !wp || !wa || !targets || !lse || !coef || !dlogits || !dh || T < 1 || H % 64 || n % 64 || n < 64 ||
      misaligned(h, 16) || misaligned(wp, 16) || misaligned(wa, 4) || misaligned(dlogits, 16) || misaligned(dh, 16))
    return set_thread_err(LS_ERR_ARG, "lsk_vocab_bwd: bad args");
  GemmCall g{};
  g.mode = ls::GEMM_FWD;
  g.A = reinterpret_cast<const bf16*>(h);
  g.lda = H;
  g.Wp = wp;
  g.force_bn = 256;
  g.g.M = T; g.g.Nw = n; g.g.Kw = H; g.g.Nout = n; g.g.Kred = H;
  g.g.absmax = wa;
  g.g.epi = ls::EPI_DLOGITS;
  g.g.out = dlogits; g.g.ldo = n;
  g.g.targets = targets; g.g.vocab_off = v0;
  g.g.lse = lse; g.g.coef = coef;
  KCK(ls::launch_nf4_gemm(g, STREAM(s)));
  KCK(gemm(ls::GEMM_DX, reinterpret_cast<const bf16*>(dlogits), n, T, wp, wa, n, H, nullptr, nullptr, 0,
           accumulate ? ls::EPI_F32_ACC : ls::EPI_F32, dh, H, nullptr, 0, STREAM(s)));
  return LS_OK;
}

int lsk_wait_flag(const uint32_t* flag, uint32_t value, int64_t limit_ns, int32_t* status, void* s) {
  if (!flag || !status || limit_ns < 0 || (reinterpret_cast<uintptr_t>(flag) & 3))
    return set_thread_err(LS_ERR_ARG, "lsk_wait_flag: bad args");
  ls::wait_flag_kernel<<<1, 32, 0, STREAM(s)>>>(flag, value, (unsigned long long)limit_ns, status);
  KLAUNCH();
  return LS_OK;
}

int lsk_device_error(int32_t* h_out, int32_t reset) {
  int v = 0;
  KCK(cudaMemcpyFromSymbol(&v, ls::g_device_error, sizeof(int)));
  if (h_out) *h_out = v;
  if (reset) {
    int z = 0;
    KCK(cudaMemcpyToSymbol(ls::g_device_error, &z, sizeof(int)));
  }
  return LS_OK;
}

}  // extern "C"
