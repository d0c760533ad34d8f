// Host side of libdflash: the C ABI, the paged KV pool and its free list, per-request
// page tables, the per-call device descriptors (staged through pinned memory), and the
// launch sequence of injection, draft step and verification.
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <functional>
#include <string>
#include <map>
#include <unordered_map>
#include <unordered_set>
#include <vector>

#include "../../include/dflash.h"
#include "kernels.h"
#include "gemm_tc.h"

using namespace dflash;

namespace {
constexpr int kPage = 64;
constexpr int kMaxSplit = 16;
constexpr int kRing = 8;

struct Stage {
  void *h = nullptr;
  void *d = nullptr;
  cudaEvent_t ev = nullptr;
  bool used = false;
};

struct Req {
  int32_t len = 0;
  std::vector<int32_t> pages;
};

int round_up(int a, int b) { return (a + b - 1) / b * b; }

// Kernel classes of the timing records.
enum KCls : int {
  K_GEMM_FC, K_GEMM_KV, K_GEMM_QKV, K_GEMM_O, K_GEMM_GATEUP, K_GEMM_DOWN, K_GEMM_LMHEAD,
  K_ATTN, K_RMSNORM, K_ROPE, K_INJECT_KV, K_SWIGLU, K_EMBED, K_TOPK, K_VERIFY, K_EXPORT, K_SAMPLE,
  K_GEMM_CONV, K_CONV, K_SELECT,
  K_NUM
};
const char *kClsName[K_NUM] = {"gemm_fc", "gemm_kv", "gemm_qkv", "gemm_o", "gemm_gateup",
                               "gemm_down", "gemm_lmhead", "attention", "rmsnorm", "qk_norm_rope",
                               "inject_kv", "swiglu", "embed", "topk", "verify", "export_kv",
                               "sample", "gemm_conv", "conv", "select"};

struct DraftGraph {
  long long key;
  int seen;
  int gen;
  int n_launch;
  cudaGraphExec_t exec;
};

struct TimeRec {
  int cls;
  cudaEvent_t a, b;
  double bytes, flops;
  int launches;
};
}  // namespace

struct dflash_ctx {
  dflash_config cfg{};
  ModelDims m{};
  int dtype = 0;
  size_t esz = 4;
  int device = 0;
  int num_sms = 0;
  dflash_weights w{};
  std::vector<dflash_layer_weights> layers;

  void *pool = nullptr;
  size_t page_elems = 0;
  std::vector<int32_t> free_pages;
  std::unordered_map<int32_t, Req> reqs;
  int max_pages_per_req = 0;
  float2 *rope = nullptr;

  // draft scratch: fp32 activations; xn, ao, hmid, xf, g are GEMM operands (fp32, or a
  // bf16 hi plane followed by a bf16 lo plane of the same row count)
  float *x = nullptr, *qkv = nullptr, *gu = nullptr;
  void *xn = nullptr, *ao = nullptr, *hmid = nullptr, *xf = nullptr;
  float *logits = nullptr, *part_o = nullptr, *part_ml = nullptr;
  int2 *cand = nullptr;    // LM-head per-tile top-k candidates [V/128][rows][topk]
  float2 *lse_part = nullptr;   // LM-head per-tile (max, sum exp) of each row [V/128][rows]
  int rows_max = 0, rows_k_max = 0;
  // injection scratch
  float *fc_out = nullptr, *kvproj = nullptr;
  void *g = nullptr;
  // sampling mode: truncated distributions of a batch's target and draft rows
  int32_t *smp_tok = nullptr, *smp_n = nullptr;
  float *smp_p = nullptr;
  // DFlash 2 modules: the convolved operand, the tap corrections [rows][2G], the
  // selector's gate rows [rows_k][r] and score tables [batch][K][topk][topk]
  void *xc = nullptr;
  float *corr = nullptr, *sel_gate = nullptr, *sel_tab = nullptr;
  // RMSNorm row statistics left by a GEMM epilogue for the next GEMM: per 128-column tile
  // and row, the sum of squares of the residual stream ([H/128][rows]; after the output
  // projection, after the down projection)
  float *ss_o = nullptr, *ss_d = nullptr;
  float *ss_inj = nullptr;   // the same after the injection's fc ([H/128][32])
  void *gath = nullptr;      // packed feature rows of dflash_inject_blocks (grown on demand)
  size_t gath_bytes = 0;
  float *ss_f = nullptr;     // and for the final norm of the K mask rows ([H/128][rows_k])

  std::vector<Stage> ring;
  size_t stage_cap = 0;
  int ring_next = 0;
  int *err_h = nullptr, *err_d = nullptr;

  TcGemm *tc = nullptr;   // tensor-core GEMM plans (bf16 only)
  AttnMaps amaps{};       // tensor maps over the KV pool for the tensor-core attention
  std::string last_error;
  int64_t launches = 0;

  // GEMM partials [S][M][N] consumed by the post-op kernels; grows on demand (never during
  // a graph capture); ws_gen counts reallocations so stale graphs are re-captured
  float *ws = nullptr;
  size_t ws_floats = 0;
  int ws_gen = 0;
  bool capturing = false;

  // CUDA graphs of the layer stack, keyed by batch size and split plan
  bool graphs_enabled = true;
  double split_overhead = 4.0;             // attention split planner: CTA overhead in pages (measured)
  std::map<std::vector<int>, int> split_cache;   // rounded page counts -> pages per split
  cudaStream_t cap_stream = nullptr;
  int32_t *desc_fixed = nullptr;   // device descriptor read by captured kernels
  std::vector<DraftGraph> graphs;

  bool timing = false;
  std::vector<TimeRec> recs;
  std::vector<cudaEvent_t> spare_events;
};

// ------------------------------------------------------------------------------ helpers
static dflash_status set_err(dflash_ctx *c, dflash_status s, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  if (c) c->last_error = buf;
  return s;
}

#define CK(ctx, expr)                                                                      \
  do {                                                                                     \
    cudaError_t e_ = (expr);                                                               \
    if (e_ != cudaSuccess)                                                                 \
      return set_err(ctx, DFLASH_ERR_CUDA, "%s failed: %s", #expr, cudaGetErrorString(e_)); \
  } while (0)

namespace {
struct DeviceGuard {
  int prev = -1;
  cudaError_t err = cudaSuccess;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
    if (prev != dev) err = cudaSetDevice(dev);
  }
  ~DeviceGuard() {
    int cur = -1;
    if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
  }
};

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }
}  // namespace

static dflash_status check_device_flag(dflash_ctx *c) {
  if (!c->err_h) return DFLASH_OK;
  int v = __atomic_exchange_n(c->err_h, 0, __ATOMIC_SEQ_CST);
  if (v) {
    const int site = __atomic_exchange_n(c->err_h + 1, 0, __ATOMIC_SEQ_CST);
    const int blk = c->err_h[2], thr = c->err_h[3], a0 = c->err_h[4], a1 = c->err_h[5];
    return set_err(c, DFLASH_ERR_DEVICE,
                   "device-side check failed earlier (code 0x%x:%s%s%s; wait site 0x%x, block "
                   "(%d,%d,%d), thread %d, progress %d/%d)",
                   v, (v & DEV_ERR_TOKEN) ? " token id out of range" : "",
                   (v & DEV_ERR_BOUNDS) ? " index out of bounds" : "",
                   (v & DEV_ERR_TIMEOUT) ? " bounded wait expired" : "", site, blk & 1023,
                   (blk >> 10) & 1023, blk >> 20, thr, a0, a1);
  }
  return DFLASH_OK;
}

static cudaEvent_t take_event(dflash_ctx *c) {
  if (!c->spare_events.empty()) {
    cudaEvent_t e = c->spare_events.back();
    c->spare_events.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

// Runs one launch (or a fixed group of launches) of kernel class `cls`; with timing on it
// is bracketed by events on its stream and tagged with its algorithmic bytes and flops.
template <typename F>
static cudaError_t timed(dflash_ctx *c, int cls, cudaStream_t s, double bytes, double flops,
                         int n_launch, F &&launch) {
  cudaEvent_t a = nullptr, b = nullptr;
  if (c->timing) {
    a = take_event(c);
    b = take_event(c);
    cudaEventRecord(a, s);
  }
  cudaError_t e = launch();
  c->launches += n_launch;
  if (c->timing) {
    cudaEventRecord(b, s);
    c->recs.push_back(TimeRec{cls, a, b, bytes, flops, n_launch});
  }
  return e;
}

static dflash_status stage_upload(dflash_ctx *c, cudaStream_t s, const void *src, size_t bytes,
                                  const int32_t **dev_out) {
  if (bytes > c->stage_cap)
    return set_err(c, DFLASH_ERR_INVALID_ARG, "descriptor of %zu bytes exceeds staging %zu", bytes,
                   c->stage_cap);
  Stage &st = c->ring[c->ring_next];
  c->ring_next = (c->ring_next + 1) % (int)c->ring.size();
  if (st.used) CK(c, cudaEventSynchronize(st.ev));
  memcpy(st.h, src, bytes);
  CK(c, cudaMemcpyAsync(st.d, st.h, bytes, cudaMemcpyHostToDevice, s));
  CK(c, cudaEventRecord(st.ev, s));
  st.used = true;
  *dev_out = (const int32_t *)st.d;
  return DFLASH_OK;
}

// Like stage_upload, into a caller-chosen device buffer.
static dflash_status stage_upload_to(dflash_ctx *c, cudaStream_t s, const void *src, size_t bytes,
                                     int32_t *dst) {
  if (bytes > c->stage_cap)
    return set_err(c, DFLASH_ERR_INVALID_ARG, "descriptor of %zu bytes exceeds staging %zu", bytes,
                   c->stage_cap);
  Stage &st = c->ring[c->ring_next];
  c->ring_next = (c->ring_next + 1) % (int)c->ring.size();
  if (st.used) CK(c, cudaEventSynchronize(st.ev));
  memcpy(st.h, src, bytes);
  CK(c, cudaMemcpyAsync(dst, st.h, bytes, cudaMemcpyHostToDevice, s));
  CK(c, cudaEventRecord(st.ev, s));
  st.used = true;
  return DFLASH_OK;
}

static dflash_status run_gemm(dflash_ctx *c, int cls, const GemmDesc &d, cudaStream_t s) {
  const double xsz = !d.x_bf16 ? 4.0 : d.x_lo2 ? 6.0 : d.x_lo[0] ? 4.0 : 2.0;
  const double out_bytes = d.epi == EPI_SWIGLU ? (double)d.M * (d.N / 2) * 4.0
                                               : (double)d.M * d.N * 4.0 * (d.epi == EPI_RESID ? 2 : 1);
  const double bytes = (double)d.N * d.K * c->esz + (double)d.M * d.K * xsz + out_bytes;
  const double flops = 2.0 * d.M * d.N * d.K;
  if (c->tc && c->dtype == DFLASH_BF16) {
    int n = tc_gemm_launches(c->tc, d);
    cudaError_t e = timed(c, cls, s, bytes, flops, n, [&] { return tc_gemm_run(c->tc, d, s); });
    if (e != cudaSuccess)
      return set_err(c, DFLASH_ERR_CUDA, "tensor-core GEMM launch failed: %s", cudaGetErrorString(e));
    return DFLASH_OK;
  }
  CK(c, timed(c, cls, s, bytes, flops, 1, [&] { return gemm_simt(c->dtype, d, s); }));
  return DFLASH_OK;
}

// Runs a GEMM in partials mode into the context workspace; *S receives the split count the
// post-op must sum.
static dflash_status gemm_ws(dflash_ctx *c, int cls, GemmDesc d, cudaStream_t s, int *S) {
  const int splits = (c->tc && c->dtype == DFLASH_BF16) ? tc_gemm_splits(c->tc, d) : 1;
  const size_t need = (size_t)splits * d.M * d.N;
  if (need > c->ws_floats) {
    if (c->capturing) return set_err(c, DFLASH_ERR_CUDA, "workspace would grow during a graph capture");
    if (c->ws) cudaFree(c->ws);
    c->ws = nullptr;
    c->ws_floats = 0;
    CK(c, cudaMalloc(&c->ws, need * sizeof(float)));
    c->ws_floats = need;
    ++c->ws_gen;
  }
  d.part = c->ws;
  *S = splits;
  return run_gemm(c, cls, d, s);
}

static GemmDesc gemm_desc(int M, int N, int K, int epi, float *y, int ldy) {
  GemmDesc d{};
  d.M = M;
  d.N = N;
  d.K = K;
  d.epi = epi;
  d.y = y;
  d.ldy = ldy;
  return d;
}

// Operand view of a scratch buffer with `rows` x `ld` elements per plane.
static OpOut op_of(const dflash_ctx *c, void *base, size_t plane_elems) {
  if (c->dtype == DFLASH_BF16) return OpOut{base, (bf16 *)base + plane_elems};
  return OpOut{base, nullptr};
}

static void set_x(const dflash_ctx *c, GemmDesc &d, const OpOut &o, int ld) {
  d.x_bf16 = c->dtype == DFLASH_BF16;
  d.n_xseg = 1;
  d.x[0] = o.hi;
  d.x_lo[0] = o.lo;
  d.x_lo2 = o.lo2;
  d.x_k0[0] = 0;
  d.x_k0[1] = d.K;
  d.ldx[0] = ld;
}

static bool fused_epilogues(const dflash_ctx *c);

static void add_wseg(GemmDesc &d, const void *w, int rows) {
  int i = d.n_wseg++;
  d.w[i] = w;
  if (i == 0) d.w_n0[0] = 0;
  d.w_n0[i + 1] = d.w_n0[i] + rows;
}

// ------------------------------------------------------------------------------ config
extern "C" dflash_status dflash_validate_config(const dflash_config *c, char *msg, int32_t msg_len) {
  auto bad = [&](dflash_status s, const char *why) {
    if (msg && msg_len > 0) snprintf(msg, (size_t)msg_len, "%s", why);
    return s;
  };
  if (!c) return bad(DFLASH_ERR_INVALID_ARG, "config is NULL");
  if (c->dtype != DFLASH_F32 && c->dtype != DFLASH_BF16) return bad(DFLASH_ERR_INVALID_ARG, "dtype");
  if (c->hidden <= 0 || c->hidden % 128 || c->hidden > 8192)
    return bad(DFLASH_ERR_UNSUPPORTED, "hidden must be a multiple of 128 in [128, 8192]");
  if (c->intermediate <= 0 || c->intermediate % 128) return bad(DFLASH_ERR_UNSUPPORTED, "intermediate must be a positive multiple of 128");
  if (c->head_dim != 64 && c->head_dim != 128) return bad(DFLASH_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
  if (c->n_q_heads <= 0 || c->n_kv_heads <= 0 || c->n_q_heads % c->n_kv_heads)
    return bad(DFLASH_ERR_INVALID_ARG, "n_q_heads must be a positive multiple of n_kv_heads");
  if (c->n_q_heads / c->n_kv_heads > 8) return bad(DFLASH_ERR_UNSUPPORTED, "GQA group above 8");
  if ((c->n_q_heads * c->head_dim) % 128 || (c->n_kv_heads * c->head_dim) % 128)
    return bad(DFLASH_ERR_UNSUPPORTED, "q and kv widths must be multiples of 128");
  if (c->n_layers < 1 || c->n_layers > 8) return bad(DFLASH_ERR_UNSUPPORTED, "n_layers must be 1..8");
  if (c->n_feat < 1 || c->n_feat > 8) return bad(DFLASH_ERR_UNSUPPORTED, "n_feat must be 1..8");
  if (c->target_hidden <= 0 || c->target_hidden % 64) return bad(DFLASH_ERR_UNSUPPORTED, "target_hidden must be a positive multiple of 64");
  if (c->block_k < 1 || c->block_k > 31) return bad(DFLASH_ERR_UNSUPPORTED, "block_k must be 1..31");
  if ((c->n_q_heads / c->n_kv_heads) * (c->block_k + 1) > 128)
    return bad(DFLASH_ERR_UNSUPPORTED, "(n_q_heads/n_kv_heads)*(block_k+1) above 128");
  if (c->vocab < 1) return bad(DFLASH_ERR_INVALID_ARG, "vocab");
  if (c->topk < 1 || c->topk > 32 || c->topk > c->vocab) return bad(DFLASH_ERR_UNSUPPORTED, "topk must be 1..min(32, vocab)");
  if (c->mask_token_id < 0 || c->mask_token_id >= c->vocab) return bad(DFLASH_ERR_INVALID_ARG, "mask_token_id out of range");
  if (c->page_size != kPage) return bad(DFLASH_ERR_UNSUPPORTED, "page_size must be 64");
  if (c->max_batch < 1 || c->max_requests < 1 || c->max_pages < 1 || c->max_inject_rows < 1)
    return bad(DFLASH_ERR_INVALID_ARG, "max_batch, max_requests, max_pages, max_inject_rows must be >= 1");
  if (c->max_positions < c->block_k + 2 || c->max_positions > (1 << 22))
    return bad(DFLASH_ERR_INVALID_ARG, "max_positions must be in [block_k + 2, 2^22]");
  if (!(c->rms_eps >= 0.f) || !(c->rope_theta > 0.f)) return bad(DFLASH_ERR_INVALID_ARG, "rms_eps / rope_theta");
  if (c->block_causal != 0 && c->block_causal != 1) return bad(DFLASH_ERR_INVALID_ARG, "block_causal must be 0 or 1");
  if (!(c->output_multiplier >= 0.f) || !(c->logit_softcap >= 0.f))
    return bad(DFLASH_ERR_INVALID_ARG, "output_multiplier and logit_softcap must be >= 0");
  if (c->dyn_conv != 0 && c->dyn_conv != 1) return bad(DFLASH_ERR_INVALID_ARG, "dyn_conv must be 0 or 1");
  if (c->selector_rank != 0 && (c->selector_rank < 32 || c->selector_rank > 512 || c->selector_rank % 32))
    return bad(DFLASH_ERR_UNSUPPORTED, "selector_rank must be 0 or a multiple of 32 in [32, 512]");
  if (msg && msg_len > 0) msg[0] = 0;
  return DFLASH_OK;
}

extern "C" const char *dflash_status_string(dflash_status s) {
  switch (s) {
    case DFLASH_OK: return "DFLASH_OK";
    case DFLASH_ERR_INVALID_ARG: return "DFLASH_ERR_INVALID_ARG";
    case DFLASH_ERR_OUT_OF_PAGES: return "DFLASH_ERR_OUT_OF_PAGES";
    case DFLASH_ERR_UNKNOWN_REQUEST: return "DFLASH_ERR_UNKNOWN_REQUEST";
    case DFLASH_ERR_CUDA: return "DFLASH_ERR_CUDA";
    case DFLASH_ERR_DEVICE: return "DFLASH_ERR_DEVICE";
    case DFLASH_ERR_UNSUPPORTED: return "DFLASH_ERR_UNSUPPORTED";
  }
  return "unknown status";
}

// ------------------------------------------------------------------------------ create / destroy
static void free_all(dflash_ctx *c) {
  void *dev[] = {c->pool, c->rope, c->x, c->xn, c->qkv, c->ao, c->gu, c->hmid, c->xf, c->logits, c->cand,
                 c->part_o, c->part_ml, c->fc_out, c->g, c->kvproj, c->smp_tok, c->smp_n, c->smp_p,
                 c->lse_part, c->xc, c->corr, c->sel_gate, c->sel_tab, c->ss_o, c->ss_d, c->ss_inj, c->ss_f, c->gath};
  for (void *p : dev)
    if (p) cudaFree(p);
  for (auto &st : c->ring) {
    if (st.h) cudaFreeHost(st.h);
    if (st.d) cudaFree(st.d);
    if (st.ev) cudaEventDestroy(st.ev);
  }
  if (c->err_h) cudaFreeHost(c->err_h);
  if (c->tc) tc_gemm_destroy(c->tc);
  for (const TimeRec &r : c->recs) {
    cudaEventDestroy(r.a);
    cudaEventDestroy(r.b);
  }
  for (cudaEvent_t e : c->spare_events) cudaEventDestroy(e);
  for (auto &g : c->graphs)
    if (g.exec) cudaGraphExecDestroy(g.exec);
  if (c->ws) cudaFree(c->ws);
  if (c->desc_fixed) cudaFree(c->desc_fixed);
  if (c->cap_stream) cudaStreamDestroy(c->cap_stream);
}

extern "C" dflash_status dflash_create(const dflash_config *cfg, const dflash_weights *w,
                                       int32_t device, dflash_ctx **out) {
  if (!out) return DFLASH_ERR_INVALID_ARG;
  *out = nullptr;
  char msg[256];
  dflash_status st = dflash_validate_config(cfg, msg, sizeof msg);
  if (st != DFLASH_OK) return st;
  if (!w || !w->embed || !w->lm_head || !w->fc || !w->fc_norm || !w->final_norm || !w->layers)
    return DFLASH_ERR_INVALID_ARG;
  const void *top[] = {w->embed, w->lm_head, w->fc, w->fc_norm, w->final_norm};
  for (const void *p : top)
    if (!aligned16(p)) return DFLASH_ERR_INVALID_ARG;
  for (int l = 0; l < cfg->n_layers; ++l) {
    const dflash_layer_weights &lw = w->layers[l];
    const void *ps[] = {lw.in_norm, lw.wq, lw.wk, lw.wv, lw.wo, lw.post_norm, lw.w_gate, lw.w_up, lw.w_down};
    for (const void *p : ps)
      if (!p || !aligned16(p)) return DFLASH_ERR_INVALID_ARG;
    if (cfg->qk_norm && (!lw.q_norm || !lw.k_norm)) return DFLASH_ERR_INVALID_ARG;
    if (cfg->dyn_conv && (!lw.conv_base || !lw.conv_proj || !aligned16(lw.conv_base) || !aligned16(lw.conv_proj)))
      return DFLASH_ERR_INVALID_ARG;
  }
  if (cfg->selector_rank) {
    const void *sel[] = {w->sel_pred_codebook, w->sel_succ_codebook, w->sel_hidden_proj};
    for (const void *p : sel)
      if (!p || !aligned16(p)) return DFLASH_ERR_INVALID_ARG;
  }

  dflash_ctx *c = new dflash_ctx();
  c->cfg = *cfg;
  c->dtype = cfg->dtype;
  c->esz = cfg->dtype == DFLASH_BF16 ? 2 : 4;
  c->device = device;
  c->w = *w;
  c->layers.assign(w->layers, w->layers + cfg->n_layers);
  c->w.layers = c->layers.data();
  ModelDims &m = c->m;
  m.H = cfg->hidden; m.L = cfg->n_layers; m.nq = cfg->n_q_heads; m.nkv = cfg->n_kv_heads;
  m.hd = cfg->head_dim; m.I = cfg->intermediate; m.V = cfg->vocab; m.K = cfg->block_k;
  m.n_feat = cfg->n_feat; m.Ht = cfg->target_hidden; m.topk = cfg->topk; m.qk_norm = cfg->qk_norm;
  m.eps = cfg->rms_eps; m.emb_scale = cfg->input_embedding_scale;
  m.causal = cfg->block_causal;
  m.out_mult = cfg->output_multiplier == 0.f ? 1.f : cfg->output_multiplier;
  m.softcap = cfg->logit_softcap;
  m.conv = cfg->dyn_conv;
  m.sel_r = cfg->selector_rank;

  auto fail = [&](dflash_status s) {
    free_all(c);
    delete c;
    return s;
  };
  DeviceGuard guard(device);
  if (guard.err != cudaSuccess) return fail(DFLASH_ERR_CUDA);
  if (cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess)
    return fail(DFLASH_ERR_CUDA);

  const size_t es = c->esz;
  const int R = cfg->max_batch * m.Q();
  const int RK = cfg->max_batch * m.K;
  const int C = cfg->max_inject_rows;
  c->rows_max = R;
  c->rows_k_max = RK;
  const size_t f4 = sizeof(float);   // an operand element takes 4 bytes (fp32, or bf16 hi + lo)
  c->page_elems = (size_t)m.L * 2 * m.nkv * kPage * m.hd;
  c->max_pages_per_req = (cfg->max_positions + kPage - 1) / kPage;
  struct Alloc { void **p; size_t bytes; } allocs[] = {
      {&c->pool, (size_t)cfg->max_pages * c->page_elems * es},
      {(void **)&c->rope, (size_t)cfg->max_positions * (m.hd / 2) * sizeof(float2)},
      {(void **)&c->x, (size_t)R * m.H * f4},
      {&c->xn, (size_t)R * m.H * f4},
      {(void **)&c->qkv, (size_t)R * m.qkv_dim() * f4},
      {&c->ao, (size_t)R * m.q_dim() * f4},
      {(void **)&c->gu, (size_t)R * 2 * m.I * f4},
      {&c->hmid, (size_t)R * m.I * f4},
      {&c->xf, (size_t)RK * m.H * f4},
      {(void **)&c->logits, (size_t)RK * m.V * f4},
      {(void **)&c->cand, (size_t)((m.V + 127) / 128) * RK * m.topk * sizeof(int2)},
      {(void **)&c->lse_part, (size_t)((m.V + 127) / 128) * RK * sizeof(float2)},
      {(void **)&c->part_o, (size_t)R * m.nq * kMaxSplit * m.hd * f4},
      {(void **)&c->part_ml, (size_t)R * m.nq * kMaxSplit * 2 * f4},
      {(void **)&c->fc_out, (size_t)C * m.H * f4},
      {&c->g, (size_t)C * m.H * (c->dtype == DFLASH_BF16 ? 6 : 4)},
      {(void **)&c->kvproj, (size_t)C * m.L * 2 * m.kv_dim() * f4},
      {(void **)&c->smp_tok, (size_t)(R + RK) * SMP_K * sizeof(int32_t)},
      {(void **)&c->smp_p, (size_t)(R + RK) * SMP_K * sizeof(float)},
      {(void **)&c->smp_n, (size_t)(R + RK) * sizeof(int32_t)},
      {&c->xc, m.conv ? (size_t)R * m.H * f4 : 0},
      {(void **)&c->corr, m.conv ? (size_t)R * 2 * (m.H / 16) * f4 : 0},
      {(void **)&c->sel_gate, (size_t)RK * m.sel_r * f4},
      {(void **)&c->sel_tab, m.sel_r ? (size_t)RK * m.topk * m.topk * f4 : 0},
      {(void **)&c->ss_o, (size_t)(m.H / 128) * R * f4},
      {(void **)&c->ss_d, (size_t)(m.H / 128) * R * f4},
      {(void **)&c->ss_inj, (size_t)(m.H / 128) * 32 * f4},
      {(void **)&c->ss_f, (size_t)(m.H / 128) * RK * f4},
  };
  for (auto &a : allocs)
    if (cudaMalloc(a.p, std::max<size_t>(a.bytes, 256)) != cudaSuccess) return fail(DFLASH_ERR_CUDA);

  // RoPE table: cos/sin(pos * theta^(-2i/hd)) evaluated in double, stored as fp32
  {
    const int half = m.hd / 2;
    std::vector<float2> tab((size_t)cfg->max_positions * half);
    for (int i = 0; i < half; ++i) {
      double inv = std::pow((double)cfg->rope_theta, -2.0 * i / m.hd);
      for (int p = 0; p < cfg->max_positions; ++p) {
        double a = (double)p * inv;
        tab[(size_t)p * half + i] = make_float2((float)std::cos(a), (float)std::sin(a));
      }
    }
    if (cudaMemcpy(c->rope, tab.data(), tab.size() * sizeof(float2), cudaMemcpyHostToDevice) != cudaSuccess)
      return fail(DFLASH_ERR_CUDA);
  }

  // every cache slot starts finite (masked positions of a page still meet a zero weight)
  if (cudaMemset(c->pool, 0, (size_t)cfg->max_pages * c->page_elems * es) != cudaSuccess)
    return fail(DFLASH_ERR_CUDA);
  c->free_pages.reserve(cfg->max_pages);
  for (int p = cfg->max_pages - 1; p >= 0; --p) c->free_pages.push_back(p);

  size_t inj = (size_t)3 * C * sizeof(int32_t);      // slot, position, source row (inject_blocks)
  size_t drf = (size_t)(4 * cfg->max_batch + 1) * sizeof(int32_t) +
               (size_t)cfg->max_batch * c->max_pages_per_req * sizeof(int32_t);
  c->stage_cap = (std::max(inj, drf) + 255) / 256 * 256;
  c->ring.resize(kRing);
  for (auto &s : c->ring) {
    if (cudaHostAlloc(&s.h, c->stage_cap, cudaHostAllocDefault) != cudaSuccess ||
        cudaMalloc(&s.d, c->stage_cap) != cudaSuccess ||
        cudaEventCreateWithFlags(&s.ev, cudaEventDisableTiming) != cudaSuccess)
      return fail(DFLASH_ERR_CUDA);
  }
  if (cudaMalloc(&c->desc_fixed, c->stage_cap) != cudaSuccess ||
      cudaStreamCreateWithFlags(&c->cap_stream, cudaStreamNonBlocking) != cudaSuccess)
    return fail(DFLASH_ERR_CUDA);
  {
    const char *ng = getenv("DFLASH_NO_GRAPHS");
    c->graphs_enabled = !(ng && ng[0] == '1');
    // per-CTA cost of the attention split kernel beyond its pages, in pages (tuning override)
    const char *so = getenv("DFLASH_SPLIT_OVERHEAD");
    if (so && so[0]) c->split_overhead = std::max(0.0, atof(so));
  }
  if (cudaHostAlloc((void **)&c->err_h, 8 * sizeof(int), cudaHostAllocMapped) != cudaSuccess ||
      cudaHostGetDevicePointer((void **)&c->err_d, c->err_h, 0) != cudaSuccess)
    return fail(DFLASH_ERR_CUDA);
  memset(c->err_h, 0, 8 * sizeof(int));

  // bf16 weights use the tensor-core GEMM; DFLASH_FORCE_FFMA=1 (diagnostics) keeps the FFMA one
  const char *force_ffma = getenv("DFLASH_FORCE_FFMA");
  if (c->dtype == DFLASH_BF16 && !(force_ffma && force_ffma[0] == '1')) {
    cudaError_t e = tc_gemm_create(&c->tc, device, c->num_sms, c->err_d);
    if (e != cudaSuccess) return fail(DFLASH_ERR_CUDA);
    if (m.hd == 128) {
      // K blocks as rows of hd values, V blocks ([hd][64]) as rows of 64 positions
      const unsigned long long blocks = (unsigned long long)cfg->max_pages * m.L * 2 * m.nkv;
      c->amaps.valid = tc_encode_2d(c->tc, c->pool, blocks * kPage, m.hd, m.hd, 64, 64, &c->amaps.k) &&
                       tc_encode_2d(c->tc, c->pool, blocks * m.hd, kPage, kPage, 64, 128, &c->amaps.v);
      c->amaps.err = c->err_d;
      c->amaps.num_sms = c->num_sms;
    }
  }
  if (cudaDeviceSynchronize() != cudaSuccess) return fail(DFLASH_ERR_CUDA);
  *out = c;
  return DFLASH_OK;
}

extern "C" void dflash_destroy(dflash_ctx *c) {
  if (!c) return;
  DeviceGuard guard(c->device);
  cudaDeviceSynchronize();
  free_all(c);
  delete c;
}

extern "C" const char *dflash_last_error(const dflash_ctx *c) { return c ? c->last_error.c_str() : ""; }
extern "C" int64_t dflash_launch_count(const dflash_ctx *c) { return c ? c->launches : 0; }
extern "C" int32_t dflash_free_pages(const dflash_ctx *c) { return c ? (int32_t)c->free_pages.size() : 0; }

extern "C" dflash_status dflash_context_len(const dflash_ctx *c, int32_t req_id, int32_t *len) {
  if (!c || !len) return DFLASH_ERR_INVALID_ARG;
  auto it = c->reqs.find(req_id);
  if (it == c->reqs.end()) return DFLASH_ERR_UNKNOWN_REQUEST;
  *len = it->second.len;
  return DFLASH_OK;
}

extern "C" dflash_status dflash_release(dflash_ctx *c, int32_t req_id) {
  if (!c) return DFLASH_ERR_INVALID_ARG;
  auto it = c->reqs.find(req_id);
  if (it == c->reqs.end()) return set_err(c, DFLASH_ERR_UNKNOWN_REQUEST, "unknown request %d", req_id);
  for (int32_t p : it->second.pages) c->free_pages.push_back(p);
  c->reqs.erase(it);
  return DFLASH_OK;
}

extern "C" dflash_status dflash_truncate(dflash_ctx *c, int32_t req_id, int32_t new_len) {
  if (!c) return DFLASH_ERR_INVALID_ARG;
  auto it = c->reqs.find(req_id);
  if (it == c->reqs.end()) return set_err(c, DFLASH_ERR_UNKNOWN_REQUEST, "unknown request %d", req_id);
  Req &r = it->second;
  if (new_len < 0 || new_len > r.len)
    return set_err(c, DFLASH_ERR_INVALID_ARG, "truncate to %d outside [0, %d]", new_len, r.len);
  size_t keep = (size_t)(new_len + kPage - 1) / kPage;
  while (r.pages.size() > keep) {
    c->free_pages.push_back(r.pages.back());
    r.pages.pop_back();
  }
  r.len = new_len;
  return DFLASH_OK;
}

// ------------------------------------------------------------------------------ injection
// block_rows == 0: the feature rows are packed (sum(n_new) of them, request after request);
// block_rows > 0: request b owns rows [b * block_rows, (b + 1) * block_rows) and its first
// n_new[b] are appended: a gather kernel packs them into library memory first, so the GEMMs
// see exactly the rows of the packed form (and take the same few-row kernels).
static dflash_status inject_impl(dflash_ctx *c, void *stream, int32_t n_req, const int32_t *req_ids,
                                 const int32_t *n_new, int32_t reset, const void *const *feats,
                                 int32_t block_rows) {
  if (!c) return DFLASH_ERR_INVALID_ARG;
  dflash_status st = check_device_flag(c);
  if (st != DFLASH_OK) return st;
  if (n_req < 0) return set_err(c, DFLASH_ERR_INVALID_ARG, "n_req < 0");
  if (n_req == 0) return DFLASH_OK;
  if (!req_ids || !n_new) return set_err(c, DFLASH_ERR_INVALID_ARG, "req_ids / n_new is NULL");
  const ModelDims &m = c->m;
  cudaStream_t s = (cudaStream_t)stream;

  // ---- plan on the host; nothing changes until every check passed
  std::unordered_set<int32_t> seen;
  long total = 0;
  int new_reqs = 0;
  long pages_needed = 0, pages_freed = 0;
  std::vector<int32_t> start(n_req);
  for (int b = 0; b < n_req; ++b) {
    if (!seen.insert(req_ids[b]).second)
      return set_err(c, DFLASH_ERR_INVALID_ARG, "request %d appears twice", req_ids[b]);
    if (n_new[b] < 0) return set_err(c, DFLASH_ERR_INVALID_ARG, "n_new[%d] < 0", b);
    if (block_rows > 0 && n_new[b] > block_rows)
      return set_err(c, DFLASH_ERR_INVALID_ARG, "n_new[%d] = %d exceeds block_rows = %d", b, n_new[b], block_rows);
    auto it = c->reqs.find(req_ids[b]);
    bool exists = it != c->reqs.end();
    if (!exists) ++new_reqs;
    int cur = (exists && !reset) ? it->second.len : 0;
    long have = (exists && !reset) ? (long)it->second.pages.size() : 0;
    if (exists && reset) pages_freed += (long)it->second.pages.size();
    long new_len = (long)cur + n_new[b];
    if (new_len + m.Q() > c->cfg.max_positions)
      return set_err(c, DFLASH_ERR_INVALID_ARG, "request %d would reach %ld positions (max %d incl. block)",
                     req_ids[b], new_len, c->cfg.max_positions);
    pages_needed += std::max(0L, (new_len + kPage - 1) / kPage - have);
    start[b] = cur;
    total += n_new[b];
  }
  if ((long)c->reqs.size() + new_reqs > c->cfg.max_requests)
    return set_err(c, DFLASH_ERR_INVALID_ARG, "more than max_requests=%d live requests", c->cfg.max_requests);
  if (pages_needed > (long)c->free_pages.size() + pages_freed)
    return set_err(c, DFLASH_ERR_OUT_OF_PAGES, "need %ld pages, %zu free", pages_needed,
                   c->free_pages.size() + (size_t)pages_freed);
  if (total > 0) {
    if (!feats) return set_err(c, DFLASH_ERR_INVALID_ARG, "feats is NULL");
    for (int f = 0; f < m.n_feat; ++f)
      if (!feats[f] || !aligned16(feats[f]))
        return set_err(c, DFLASH_ERR_INVALID_ARG, "feats[%d] is NULL or not 16-byte aligned", f);
  }
  DeviceGuard guard(c->device);
  if (guard.err != cudaSuccess) return set_err(c, DFLASH_ERR_CUDA, "cudaSetDevice failed");

  const int C = c->cfg.max_inject_rows;
  const size_t row_bytes = (size_t)m.Ht * c->esz;
  if (block_rows > 0 && total > 0) {
    const size_t need = (size_t)m.n_feat * (size_t)std::min<long>(C, total) * row_bytes;
    if (need > c->gath_bytes) {
      if (c->gath) cudaFree(c->gath);
      c->gath = nullptr;
      c->gath_bytes = 0;
      if (cudaMalloc(&c->gath, need) != cudaSuccess) {
        cudaGetLastError();
        return set_err(c, DFLASH_ERR_CUDA, "cudaMalloc of %zu bytes for the packed feature rows failed", need);
      }
      c->gath_bytes = need;
    }
  }

  // ---- commit: pages and lengths
  std::vector<int32_t> slot(total), pos(total), src(block_rows > 0 ? total : 0);
  long r = 0;
  for (int b = 0; b < n_req; ++b) {
    Req &q = c->reqs[req_ids[b]];
    if (reset) {
      for (int32_t p : q.pages) c->free_pages.push_back(p);
      q.pages.clear();
      q.len = 0;
    }
    int new_len = start[b] + n_new[b];
    while ((int)q.pages.size() * kPage < new_len) {
      q.pages.push_back(c->free_pages.back());
      c->free_pages.pop_back();
    }
    for (int i = 0; i < n_new[b]; ++i, ++r) {
      int p = start[b] + i;
      slot[r] = q.pages[p / kPage] * kPage + p % kPage;
      pos[r] = p;
      if (block_rows > 0) src[r] = b * block_rows + i;
    }
    q.len = new_len;
  }

  // ---- launches, in chunks of max_inject_rows rows
  const int F = m.n_feat * m.Ht;
  const int kvw = m.L * 2 * m.kv_dim();
  std::vector<int32_t> buf;
  std::vector<const void *> knorm(m.L);
  for (int l = 0; l < m.L; ++l) knorm[l] = c->layers[l].k_norm;
  for (long r0 = 0; r0 < total; r0 += C) {
    int n = (int)std::min<long>(C, total - r0);
    buf.assign(slot.begin() + r0, slot.begin() + r0 + n);
    buf.insert(buf.end(), pos.begin() + r0, pos.begin() + r0 + n);
    if (block_rows > 0) buf.insert(buf.end(), src.begin() + r0, src.begin() + r0 + n);
    const int32_t *dslot = nullptr;
    if ((st = stage_upload(c, s, buf.data(), buf.size() * 4, &dslot)) != DFLASH_OK) return st;
    // the feature rows of this chunk: read in place, or the counted rows of the blocks packed
    const void *fx[8];
    for (int f = 0; f < m.n_feat; ++f)
      fx[f] = block_rows > 0 ? (const void *)((const char *)c->gath + (size_t)f * n * row_bytes)
                             : (const void *)((const char *)feats[f] + (size_t)r0 * row_bytes);
    if (block_rows > 0)
      CK(c, timed(c, K_INJECT_KV, s, 2.0 * n * m.n_feat * row_bytes, 0, 1, [&] {
           return launch_gather_rows(m.n_feat, n, (long)row_bytes, dslot + 2 * n, feats, c->gath,
                                     (long)n * (long)row_bytes, s);
         }));
    // fc over the n_feat feature tensors read in place (K segments), then RMSNorm -> g
    GemmDesc d = gemm_desc(n, m.H, F, EPI_STORE, nullptr, m.H);
    d.x_bf16 = c->dtype == DFLASH_BF16;   // the features are exact storage-type values
    d.n_xseg = m.n_feat;
    for (int f = 0; f < m.n_feat; ++f) {
      d.x[f] = fx[f];
      d.x_k0[f] = f * m.Ht;
      d.ldx[f] = m.Ht;
    }
    d.x_k0[m.n_feat] = F;
    add_wseg(d, c->w.fc, m.H);
    d.exact_acc = 1;                      // g decides how the cached K/V round
    int S = 1;
    OpOut g = op_of(c, c->g, (size_t)C * m.H);
    if (g.lo) g.lo2 = (bf16 *)g.lo + (size_t)C * m.H;   // g carries three planes
    // few rows on the tensor cores: the fc epilogue writes fc_out * fc_norm and its per-tile
    // sums of squares, and the K/V GEMM applies the RMSNorm row scale (one launch fewer)
    const bool fnorm = c->tc && c->dtype == DFLASH_BF16 && n <= 32;
    if (fnorm) {
      d.epi = EPI_RESNORM;
      d.out = g;
      d.ldo = m.H;
      d.norm_w = c->w.fc_norm;
      d.ss_part = c->ss_inj;
      if ((st = run_gemm(c, K_GEMM_FC, d, s)) != DFLASH_OK) return st;
    } else {
      if ((st = gemm_ws(c, K_GEMM_FC, d, s, &S)) != DFLASH_OK) return st;
      CK(c, timed(c, K_RMSNORM, s, 4.0 * n * m.H * (S + 1), 4.0 * n * m.H, 1, [&] {
           return launch_post_norm(c->dtype, n, m.H, c->ws, S, nullptr, g, c->w.fc_norm, m.eps, 0, s);
         }));
    }
    // every layer's [Wk; Wv] in one GEMM, then k-norm + RoPE + paged write
    GemmDesc e = gemm_desc(n, kvw, m.H, EPI_STORE, nullptr, kvw);
    set_x(c, e, g, m.H);
    e.exact_acc = 1;                      // rounded to the storage type in the cache
    if (fnorm) {
      e.rs_part = c->ss_inj;
      e.rs_tiles = m.H / 128;
      e.rs_dim = m.H;
      e.eps = m.eps;
    }
    for (int l = 0; l < m.L; ++l) {
      add_wseg(e, c->layers[l].wk, m.kv_dim());
      add_wseg(e, c->layers[l].wv, m.kv_dim());
    }
    if (fnorm && fused_epilogues(c) && m.L <= 8) {
      // ... and its epilogue does the k-norm, RoPE and paged-cache write (one head per tile)
      e.epi = EPI_KVCACHE;
      e.kv_slot = dslot;
      e.kv_pos = dslot + n;
      e.kv_pool = c->pool;
      for (int l = 0; l < m.L; ++l) e.kv_knorm[l] = m.qk_norm ? c->layers[l].k_norm : nullptr;
      e.kv_L = m.L;
      e.kv_nkv = m.nkv;
      e.kv_dim = m.kv_dim();
      e.rope = c->rope;
      if ((st = run_gemm(c, K_GEMM_KV, e, s)) != DFLASH_OK) return st;
      continue;
    }
    if ((st = gemm_ws(c, K_GEMM_KV, e, s, &S)) != DFLASH_OK) return st;
    CK(c, timed(c, K_INJECT_KV, s, (double)n * kvw * (4.0 * S + c->esz), 8.0 * n * kvw, 1, [&] {
         return launch_post_kv(c->dtype, m, n, c->ws, S, dslot, dslot + n, c->rope, knorm.data(),
                               c->pool, s);
       }));
  }
  return DFLASH_OK;
}

extern "C" dflash_status dflash_inject_context(dflash_ctx *c, void *stream, int32_t n_req,
                                               const int32_t *req_ids, const int32_t *n_new,
                                               int32_t reset, const void *const *feats) {
  return inject_impl(c, stream, n_req, req_ids, n_new, reset, feats, 0);
}

extern "C" dflash_status dflash_inject_blocks(dflash_ctx *c, void *stream, int32_t n_req,
                                              const int32_t *req_ids, const int32_t *n_new,
                                              int32_t block_rows, const void *const *feats) {
  if (c && block_rows < 1) return set_err(c, DFLASH_ERR_INVALID_ARG, "block_rows < 1");
  if (c && (long)n_req * block_rows > 0x7fffffffL)
    return set_err(c, DFLASH_ERR_INVALID_ARG, "n_req * block_rows exceeds 2^31 - 1 feature rows");
  return inject_impl(c, stream, n_req, req_ids, n_new, 0, feats, block_rows);
}

// ------------------------------------------------------------------------------ draft step
// Context splits of a batch. Every request's context is cut into chunks of P whole pages
// (its last chunk shorter), so long contexts get more splits than short ones. The CTA of a
// (split, kv head, request) costs its pages plus a fixed setup and epilogue overhead, and
// the block scheduler hands CTAs to free SMs in launch order (split fastest, request
// slowest): the layer's attention time is the makespan of that list schedule on `slots`
// resident CTAs. P is the candidate, from the longest context cut into 1..kMaxSplit
// chunks, with the smallest simulated makespan; a finer cut must win by 2% to be taken.
static int choose_split_pages(const std::vector<int> &pages, int nkv, int slots, double ovh, int tile) {
  const int B = (int)pages.size();
  int maxp = 0;
  for (int b = 0; b < B; ++b) maxp = std::max(maxp, pages[b]);
  int best_P = maxp, prev_P = -1;
  double best = 0;
  std::vector<double> heap;
  for (int k = 1; k <= kMaxSplit; ++k) {
    // whole tiles of `tile` pages per split (the tensor-core kernel takes two pages a tile)
    const int P = ((maxp + k - 1) / k + tile - 1) / tile * tile;
    if (P == prev_P) continue;
    prev_P = P;
    long n_cta = 0;
    for (int b = 0; b < B; ++b) n_cta += (long)nkv * ((pages[b] + P - 1) / P);
    if (k > 1 && n_cta > 8L * slots) break;      // finer cuts only add CTAs from here
    heap.assign(slots, 0.0);                     // min-heap of slot free times
    double span = 0;
    for (int b = 0; b < B; ++b) {
      const int ns = (pages[b] + P - 1) / P;
      for (int h = 0; h < nkv; ++h)
        for (int sp = 0; sp < ns; ++sp) {
          std::pop_heap(heap.begin(), heap.end(), std::greater<double>());
          const int len = std::min(P, pages[b] - sp * P);
          const double t = heap.back() + (len + tile - 1) / tile * tile + ovh;
          heap.back() = t;
          std::push_heap(heap.begin(), heap.end(), std::greater<double>());
          span = std::max(span, t);
        }
    }
    if (k == 1 || span < 0.98 * best) {
      best = span;
      best_P = P;
    }
  }
  return best_P;
}

// The split plan of a batch. The simulation above costs ~0.3 ms of host time for 8 requests
// of 512 pages; it runs on page counts rounded up to 8 pages, and its choice is remembered
// per rounded batch, so a batch whose contexts grow by a few positions per step (or come
// back to the same lengths) reuses it. Any split length is a valid plan (the last split of a
// request is shorter); the rounding only shifts which one the heuristic picks.
static void plan_splits(dflash_ctx *c, const std::vector<int> &pages, int nkv, int slots, double ovh, int tile,
                        std::vector<int> &n_split, std::vector<int> &split_len) {
  const int B = (int)pages.size();
  n_split.assign(B, 0);
  split_len.assign(B, kPage);
  int maxp = 0;
  std::vector<int> key(B + 3);
  for (int b = 0; b < B; ++b) {
    maxp = std::max(maxp, pages[b]);
    key[b] = (pages[b] + 7) / 8 * 8;
  }
  if (maxp == 0) return;
  key[B] = nkv;
  key[B + 1] = slots;
  key[B + 2] = tile;
  int P;
  auto it = c->split_cache.find(key);
  if (it != c->split_cache.end()) {
    P = it->second;
  } else {
    std::vector<int> rounded(key.begin(), key.begin() + B);
    P = choose_split_pages(rounded, nkv, slots, ovh, tile);
    if (c->split_cache.size() >= 1024) c->split_cache.clear();
    c->split_cache.emplace(std::move(key), P);
  }
  for (int b = 0; b < B; ++b) {
    n_split[b] = (pages[b] + P - 1) / P;
    split_len[b] = P * kPage;
  }
}

// The LM head ranks candidates inside the tensor-core GEMM epilogue while the token tile is
// narrow (at most 32 rows: a few selection rounds per warp); wider tiles write the fp32
// logits and rank them row by row, which is cheaper than 32+ rounds per warp per tile.
static bool fused_topk(const dflash_ctx *c, int rows) { return c->tc && rows <= 32; }

// q/k norm + RoPE and SwiGLU run in the tensor-core GEMM epilogues when a head is one
// 128-row weight tile; otherwise (FFMA GEMM, head_dim 64) they are separate post-ops.
// Whether a step of R block rows defers its RMSNorms to the next GEMM (the residual add in
// the output / down projection epilogues, the row scale applied by the consumer). The final
// norm's operand xf then holds x * w_final, and every GEMM that reads it (the LM head, the
// selector's gate) takes the row scale from ss_f.
static bool fused_norms(const dflash_ctx *c, int R) {
  return fused_epilogues(c) && !c->m.conv && c->m.I % 64 == 0 && R <= 32;
}

static bool fused_epilogues(const dflash_ctx *c) {
  return c->tc && c->m.hd == 128 && c->m.q_dim() % 128 == 0 && c->m.kv_dim() % 128 == 0;
}

// The layer stack of the draft step plus the final norm and the LM-head GEMM: every launch
// between the embedding and the top-k selection. It touches only library buffers and the
// device descriptor `bt`, so it can be captured once per (batch, split plan) and replayed.
static dflash_status draft_layers(dflash_ctx *c, int B, const DraftBatch &bt, double attn_bytes,
                                  double attn_flops, float *logits, cudaStream_t s) {
  const ModelDims &m = c->m;
  dflash_status st;
  const int R = B * m.Q(), RK = B * m.K;
  const OpOut xn = op_of(c, c->xn, (size_t)c->rows_max * m.H);
  const OpOut ao = op_of(c, c->ao, (size_t)c->rows_max * m.q_dim());
  const OpOut hm = op_of(c, c->hmid, (size_t)c->rows_max * m.I);
  const OpOut xf = op_of(c, c->xf, (size_t)c->rows_k_max * m.H);
  // DFlash 2 convolutions: the tap corrections come from a GEMM over the convolution's
  // input rows; xc holds the convolved operand (input side) or the sublayer output as an
  // operand (output side)
  const OpOut xc = op_of(c, c->xc, (size_t)c->rows_max * m.H);
  const int G2 = 2 * (m.H / 16);
  auto conv_taps = [&](const dflash_layer_weights &lw, int j, const void **base) -> dflash_status {
    *base = (const char *)lw.conv_base + (size_t)j * 2 * m.H * c->esz;
    const void *proj = (const char *)lw.conv_proj + (size_t)j * G2 * m.H * c->esz;
    GemmDesc d = gemm_desc(R, G2, m.H, EPI_STORE, c->corr, G2);
    set_x(c, d, j % 2 ? xc : xn, m.H);
    add_wseg(d, proj, G2);
    return run_gemm(c, K_GEMM_CONV, d, s);
  };
  auto conv_in = [&](const dflash_layer_weights &lw, int j) -> dflash_status {
    const void *base;
    dflash_status e = conv_taps(lw, j, &base);
    if (e != DFLASH_OK) return e;
    CK(c, timed(c, K_CONV, s, (double)R * m.H * 12 + (double)R * G2 * 4, 4.0 * R * m.H, 1, [&] {
         return launch_conv_in(c->dtype, R, m.Q(), m.H, xn, c->corr, base, xc, s);
       }));
    return DFLASH_OK;
  };
  // output side: the GEMM product in ws -> operand -> taps -> x += conv, next norm
  auto conv_out = [&](const dflash_layer_weights &lw, int j, int S_, OpOut out, const void *nw,
                      int skip) -> dflash_status {
    if (S_ != 1) return set_err(c, DFLASH_ERR_CUDA, "convolution after a split GEMM product");
    CK(c, timed(c, K_CONV, s, (double)R * m.H * 8, 0.0, 1,
                [&] { return launch_to_op((long)R * m.H, c->ws, xc, s); }));
    const void *base;
    dflash_status e = conv_taps(lw, j, &base);
    if (e != DFLASH_OK) return e;
    CK(c, timed(c, K_CONV, s, (double)R * m.H * 20 + (double)R * G2 * 4, 8.0 * R * m.H, 1, [&] {
         return launch_conv_out_norm(c->dtype, R, m.Q(), m.H, c->ws, c->corr, base, c->x, out, nw, m.eps,
                                     skip, s);
       }));
    return DFLASH_OK;
  };
  // tensor-core path with few rows: the residual add runs in the output / down projection's
  // epilogue, which also writes x * w (w the next RMSNorm's weight) as the next GEMM's
  // operand and each 128-column tile's sum of squares per row; the next GEMM scales its
  // rows by the RMSNorm factor. This saves two dependent launches per layer, which is what
  // a batch-1 step is made of; with more rows the epilogue's per-token residual loads cost
  // more than the launches (measured), and the row kernel stays. The last layer's final
  // norm is always the row kernel (it feeds the LM head the K mask rows only).
  const bool fnorm = fused_norms(c, R);
  auto rs_from = [&](GemmDesc &d, const float *ss) {
    d.rs_part = ss;
    d.rs_tiles = m.H / 128;
    d.rs_dim = m.H;
    d.eps = m.eps;
  };
  int S = 1;
  for (int l = 0; l < m.L; ++l) {
    const dflash_layer_weights &lw = c->layers[l];
    if (m.conv && (st = conv_in(lw, 0)) != DFLASH_OK) return st;
    // q/k/v projection with per-head q/k norm + RoPE: in the tensor-core GEMM's epilogue
    // (one 128-wide head per tile), else as a post-op
    GemmDesc d = gemm_desc(R, m.qkv_dim(), m.H, EPI_STORE, nullptr, m.qkv_dim());
    set_x(c, d, m.conv ? xc : xn, m.H);
    add_wseg(d, lw.wq, m.q_dim());
    add_wseg(d, lw.wk, m.kv_dim());
    add_wseg(d, lw.wv, m.kv_dim());
    if (fused_epilogues(c)) {
      d.epi = EPI_QKV;
      d.y = c->qkv;
      d.ctx_len = bt.ctx_len;
      d.rope = c->rope;
      d.q_norm = m.qk_norm ? lw.q_norm : nullptr;
      d.k_norm = m.qk_norm ? lw.k_norm : nullptr;
      d.eps = m.eps;
      d.rows_per_req = m.Q();
      d.q_dim = m.q_dim();
      d.kv_dim = m.kv_dim();
      if (fnorm && l > 0) rs_from(d, c->ss_d);     // layer 0's input comes normalised
      if ((st = run_gemm(c, K_GEMM_QKV, d, s)) != DFLASH_OK) return st;
    } else {
      if ((st = gemm_ws(c, K_GEMM_QKV, d, s, &S)) != DFLASH_OK) return st;
      CK(c, timed(c, K_ROPE, s, 4.0 * R * m.qkv_dim() * (S + 1), 8.0 * R * (m.nq + m.nkv) * m.hd, 1, [&] {
           return launch_post_qkv(c->dtype, m, B, c->ws, S, c->qkv, bt.ctx_len, c->rope, lw.q_norm,
                                  lw.k_norm, s);
         }));
    }
    const int attn_launches = bt.max_split == 0 ? 1 : 2;     // the split kernel, then the combine
    CK(c, timed(c, K_ATTN, s, attn_bytes, attn_flops, attn_launches, [&] {
         return launch_attention(c->dtype, m, bt, l, c->qkv, c->pool, c->part_o, c->part_ml, ao,
                                 c->amaps.valid ? &c->amaps : nullptr, s);
       }));
    // output projection; post-op: residual add + post-attention norm
    GemmDesc o = gemm_desc(R, m.H, m.q_dim(), EPI_STORE, nullptr, m.H);
    set_x(c, o, ao, m.q_dim());
    add_wseg(o, lw.wo, m.H);
    if (fnorm) {
      o.epi = EPI_RESNORM;
      o.y = c->x;
      o.out = xn;
      o.ldo = m.H;
      o.norm_w = lw.post_norm;
      o.ss_part = c->ss_o;
      if ((st = run_gemm(c, K_GEMM_O, o, s)) != DFLASH_OK) return st;
    } else if ((st = gemm_ws(c, K_GEMM_O, o, s, &S)) != DFLASH_OK) {
      return st;
    }
    if (m.conv) {
      if ((st = conv_out(lw, 1, S, xn, lw.post_norm, 0)) != DFLASH_OK) return st;
      if ((st = conv_in(lw, 2)) != DFLASH_OK) return st;
    } else if (!fnorm) {
      CK(c, timed(c, K_RMSNORM, s, 4.0 * R * m.H * (S + 3), 4.0 * R * m.H, 1, [&] {
           return launch_post_norm(c->dtype, R, m.H, c->ws, S, c->x, xn, lw.post_norm, m.eps, 0, s);
         }));
    }
    // gate/up projection with SwiGLU: in the tensor-core GEMM's epilogue (a tile takes 64
    // gate and the same 64 up rows), else as a post-op
    GemmDesc gu = gemm_desc(R, 2 * m.I, m.H, EPI_STORE, nullptr, 2 * m.I);
    set_x(c, gu, m.conv ? xc : xn, m.H);
    add_wseg(gu, lw.w_gate, m.I);
    add_wseg(gu, lw.w_up, m.I);
    if (fused_epilogues(c) && m.I % 64 == 0) {
      gu.epi = EPI_SWIGLU;
      gu.out = hm;
      gu.ldo = m.I;
      if (fnorm) rs_from(gu, c->ss_o);
      if ((st = run_gemm(c, K_GEMM_GATEUP, gu, s)) != DFLASH_OK) return st;
    } else {
      if ((st = gemm_ws(c, K_GEMM_GATEUP, gu, s, &S)) != DFLASH_OK) return st;
      CK(c, timed(c, K_SWIGLU, s, 4.0 * R * m.I * (2 * S + 1), 5.0 * R * m.I, 1,
                  [&] { return launch_post_swiglu(R, m.I, c->ws, S, hm, s); }));
    }
    // down projection; post-op: residual add + the next layer's input norm, or after the
    // last layer the final norm of the K mask rows (the anchor row yields no candidate)
    GemmDesc dn = gemm_desc(R, m.H, m.I, EPI_STORE, nullptr, m.H);
    set_x(c, dn, hm, m.I);
    add_wseg(dn, lw.w_down, m.H);
    const bool last = l + 1 == m.L;
    const void *nw = last ? c->w.final_norm : c->layers[l + 1].in_norm;
    if (fnorm) {
      // the last layer leaves the final norm's operand (K mask rows only) and sums for the
      // LM head
      dn.epi = EPI_RESNORM;
      dn.y = c->x;
      dn.out = last ? xf : xn;
      dn.ldo = m.H;
      dn.norm_w = nw;
      dn.ss_part = last ? c->ss_f : c->ss_d;
      dn.out_skip_k = last ? m.K : 0;
      if ((st = run_gemm(c, K_GEMM_DOWN, dn, s)) != DFLASH_OK) return st;
      continue;
    }
    if ((st = gemm_ws(c, K_GEMM_DOWN, dn, s, &S)) != DFLASH_OK) return st;
    if (m.conv) {
      if ((st = conv_out(lw, 3, S, last ? xf : xn, nw, last ? m.K : 0)) != DFLASH_OK) return st;
    } else {
      CK(c, timed(c, K_RMSNORM, s, 4.0 * R * m.H * (S + 3), 4.0 * R * m.H, 1, [&] {
           return launch_post_norm(c->dtype, R, m.H, c->ws, S, c->x, last ? xf : xn, nw, m.eps,
                                   last ? m.K : 0, s);
         }));
    }
  }
  if (fused_topk(c, RK)) {
    // tensor-core LM head: per-tile top-k in the GEMM epilogue (merged afterwards); full
    // logits are written only when the caller asks for them
    GemmDesc lm = gemm_desc(RK, m.V, m.H, EPI_TOPK, logits, m.V);
    set_x(c, lm, xf, m.H);
    add_wseg(lm, c->w.lm_head, m.V);
    lm.topk = m.topk;
    lm.cand = c->cand;
    lm.lse_part = c->lse_part;
    lm.out_xf = m.out_mult != 1.f || m.softcap > 0.f;
    lm.out_mult = m.out_mult;
    lm.out_cap = m.softcap;
    if (fnorm) rs_from(lm, c->ss_f);
    if ((st = run_gemm(c, K_GEMM_LMHEAD, lm, s)) != DFLASH_OK) return st;
  } else {
    float *lg = logits ? logits : c->logits;
    GemmDesc lm = gemm_desc(RK, m.V, m.H, EPI_STORE, lg, m.V);
    set_x(c, lm, xf, m.H);
    add_wseg(lm, c->w.lm_head, m.V);
    if ((st = run_gemm(c, K_GEMM_LMHEAD, lm, s)) != DFLASH_OK) return st;
    if (m.out_mult != 1.f || m.softcap > 0.f)
      CK(c, timed(c, K_TOPK, s, 8.0 * RK * m.V, 4.0 * RK * m.V, 1,
                  [&] { return launch_logit_xform((long)RK * m.V, m.out_mult, m.softcap, lg, s); }));
  }
  return DFLASH_OK;
}

// Replays (or, on the second sighting of this batch size and split plan, captures) the
// layer stack as a CUDA graph. Capture runs on the library's own stream (captures never
// execute); the graph is launched on the caller's stream.
static dflash_status run_layers_graph(dflash_ctx *c, int B, const DraftBatch &bt, cudaStream_t s) {
  // the batch size and the split plan select the graph
  const long long key = ((long long)B << 8) | bt.max_split;
  const int gen = tc_gemm_generation(c->tc) * 4096 + c->ws_gen;
  for (auto &g : c->graphs) {
    if (g.key != key) continue;
    if (g.exec && g.gen == gen) {
      CK(c, cudaGraphLaunch(g.exec, s));
      c->launches += g.n_launch;
      return DFLASH_OK;
    }
    if (g.exec) {                       // a GEMM workspace moved since the capture
      cudaGraphExecDestroy(g.exec);
      g.exec = nullptr;
    }
    if (g.seen++ < 1) break;            // run eagerly until the plan has been seen twice
    const int64_t l0 = c->launches;
    CK(c, cudaStreamBeginCapture(c->cap_stream, cudaStreamCaptureModeThreadLocal));
    c->capturing = true;
    dflash_status st = draft_layers(c, B, bt, 0, 0, nullptr, c->cap_stream);
    c->capturing = false;
    cudaGraph_t graph = nullptr;
    cudaError_t e = cudaStreamEndCapture(c->cap_stream, &graph);
    c->launches = l0;
    if (st != DFLASH_OK) {
      if (graph) cudaGraphDestroy(graph);
      return st;
    }
    if (e != cudaSuccess) return set_err(c, DFLASH_ERR_CUDA, "graph capture: %s", cudaGetErrorString(e));
    size_t n_nodes = 0;
    cudaGraphGetNodes(graph, nullptr, &n_nodes);
    e = cudaGraphInstantiate(&g.exec, graph, 0);
    cudaGraphDestroy(graph);
    if (e != cudaSuccess) {
      g.exec = nullptr;
      return set_err(c, DFLASH_ERR_CUDA, "graph instantiate: %s", cudaGetErrorString(e));
    }
    g.gen = gen;
    g.n_launch = (int)n_nodes;
    CK(c, cudaGraphLaunch(g.exec, s));
    c->launches += g.n_launch;
    return DFLASH_OK;
  }
  bool found = false;
  for (auto &g : c->graphs) found |= g.key == key;
  if (!found) {
    if (c->graphs.size() >= 16) {
      if (c->graphs.front().exec) cudaGraphExecDestroy(c->graphs.front().exec);
      c->graphs.erase(c->graphs.begin());
    }
    c->graphs.push_back(DraftGraph{key, 1, gen, 0, nullptr});
  }
  return draft_layers(c, B, bt, 0, 0, nullptr, s);
}

static dflash_status draft_step_impl(dflash_ctx *c, void *stream, int32_t n_req,
                                     const int32_t *req_ids, const int32_t *anchors, int32_t *argmax,
                                     int32_t *topk_idx, float *topk_val, float *logits, float *lse,
                                     int32_t *selected = nullptr, const SelSample *sel_smp = nullptr) {
  if (!c) return DFLASH_ERR_INVALID_ARG;
  dflash_status st = check_device_flag(c);
  if (st != DFLASH_OK) return st;
  if (n_req < 1 || n_req > c->cfg.max_batch)
    return set_err(c, DFLASH_ERR_INVALID_ARG, "n_req=%d outside [1, max_batch=%d]", n_req, c->cfg.max_batch);
  if (!req_ids || !anchors || !argmax) return set_err(c, DFLASH_ERR_INVALID_ARG, "NULL argument");
  if ((topk_idx == nullptr) != (topk_val == nullptr))
    return set_err(c, DFLASH_ERR_INVALID_ARG, "topk_idx and topk_val must both be given or both NULL");
  if (selected && (!c->m.sel_r || !topk_idx))
    return set_err(c, DFLASH_ERR_INVALID_ARG, "selected needs selector_rank > 0 and the top-k outputs");
  const ModelDims &m = c->m;
  const int B = n_req, Q = m.Q();
  std::vector<int32_t> desc(4 * B + 1);
  std::vector<const Req *> rq(B);
  std::unordered_set<int32_t> seen;
  int max_split = 0;
  std::vector<int> pages(B), ns, sl;
  for (int b = 0; b < B; ++b) {
    if (!seen.insert(req_ids[b]).second)
      return set_err(c, DFLASH_ERR_INVALID_ARG, "request %d appears twice", req_ids[b]);
    auto it = c->reqs.find(req_ids[b]);
    if (it == c->reqs.end()) return set_err(c, DFLASH_ERR_UNKNOWN_REQUEST, "unknown request %d", req_ids[b]);
    rq[b] = &it->second;
    pages[b] = (rq[b]->len + kPage - 1) / kPage;
  }
  // the tensor-core split kernel runs one CTA per SM, the FFMA one two
  const bool attn_tc = c->amaps.valid;
  plan_splits(c, pages, m.nkv, (attn_tc ? 1 : 2) * c->num_sms, c->split_overhead, attn_tc ? 2 : 1, ns, sl);
  for (int b = 0; b < B; ++b) {
    desc[b] = rq[b]->len;
    desc[B + b] = ns[b];
    desc[2 * B + b] = sl[b];
    max_split = std::max(max_split, ns[b]);
  }
  int off = 0;
  for (int b = 0; b < B; ++b) {
    desc[3 * B + b] = off;
    off += (int)rq[b]->pages.size();
  }
  desc[4 * B] = off;
  for (int b = 0; b < B; ++b) desc.insert(desc.end(), rq[b]->pages.begin(), rq[b]->pages.end());

  // algorithmic work of one layer's attention: read every context K/V once, 4 flops per
  // (query row, head, dim, key) for scores and the weighted sum
  double attn_bytes = 0, attn_flops = 0;
  for (int b = 0; b < B; ++b) {
    double S = (double)rq[b]->len + Q;
    attn_bytes += (double)rq[b]->len * 2 * m.kv_dim() * c->esz + (double)Q * (m.q_dim() + 2 * m.kv_dim()) * 4 +
                  (double)Q * m.q_dim() * 4;
    attn_flops += 4.0 * Q * m.nq * m.hd * S;
  }
  DeviceGuard guard(c->device);
  if (guard.err != cudaSuccess) return set_err(c, DFLASH_ERR_CUDA, "cudaSetDevice failed");
  cudaStream_t s = (cudaStream_t)stream;
  const int RK = B * m.K;
  const bool use_graph = c->tc && !logits && !c->timing && c->graphs_enabled;
  const int32_t *dd = nullptr;
  if (use_graph) {
    // the descriptor goes to a fixed device buffer that the captured kernels read
    if ((st = stage_upload_to(c, s, desc.data(), desc.size() * 4, c->desc_fixed)) != DFLASH_OK) return st;
    dd = c->desc_fixed;
  } else if ((st = stage_upload(c, s, desc.data(), desc.size() * 4, &dd)) != DFLASH_OK) {
    return st;
  }
  DraftBatch bt{dd, dd + B, dd + 2 * B, dd + 3 * B, dd + 4 * B + 1, B, max_split,
                *std::min_element(ns.begin(), ns.end())};

  // block embedding [anchor, mask x K] x scale, fused with the first layer's input norm
  const OpOut xn0 = op_of(c, c->xn, (size_t)c->rows_max * m.H);
  CK(c, timed(c, K_EMBED, s, (double)B * Q * m.H * (c->esz + 8), (double)B * Q * m.H * 4, 1, [&] {
       return launch_embed_norm(c->dtype, m, B, anchors, c->cfg.mask_token_id, c->w.embed,
                                c->w.mask_embedding, c->x, xn0, c->layers[0].in_norm, c->err_d, s);
     }));
  if (use_graph) {
    if ((st = run_layers_graph(c, B, bt, s)) != DFLASH_OK) return st;
  } else if ((st = draft_layers(c, B, bt, attn_bytes, attn_flops, logits, s)) != DFLASH_OK) {
    return st;
  }
  if (fused_topk(c, RK)) {
    const int tiles = (m.V + 127) / 128;
    CK(c, timed(c, K_TOPK, s, 8.0 * tiles * RK * m.topk, 1.0 * tiles * RK * m.topk, 1, [&] {
         return launch_topk_merge(tiles, RK, m.topk, c->cand, argmax, topk_idx, topk_val, c->lse_part, lse, s);
       }));
  } else {
    float *lg = logits ? logits : c->logits;
    CK(c, timed(c, K_TOPK, s, 4.0 * RK * m.V, 1.0 * RK * m.V, 1, [&] {
         return launch_topk(RK, m.V, m.topk, lg, argmax, topk_idx, topk_val, lse, 0, s);
       }));
  }
  if (selected) {
    // path selector: gate rows g_t = W_h h_t from the final-normed rows, then the score
    // tables and the walk
    const int r = m.sel_r;
    GemmDesc gd = gemm_desc(RK, r, m.H, EPI_STORE, c->sel_gate, r);
    set_x(c, gd, op_of(c, c->xf, (size_t)c->rows_k_max * m.H), m.H);
    add_wseg(gd, c->w.sel_hidden_proj, r);
    if (fused_norms(c, B * Q)) {          // xf holds x * w_final: apply the norm's row scale
      gd.rs_part = c->ss_f;
      gd.rs_tiles = m.H / 128;
      gd.rs_dim = m.H;
      gd.eps = m.eps;
    }
    if ((st = run_gemm(c, K_SELECT, gd, s)) != DFLASH_OK) return st;
    const double rows = (double)RK * m.topk * 2 + B;
    CK(c, timed(c, K_SELECT, s, rows * r * c->esz + (double)RK * r * 4, 2.0 * RK * m.topk * m.topk * r, 2, [&] {
         return launch_select_path(c->dtype, B, m.K, m.topk, r, m.V, anchors, topk_idx, topk_val, c->sel_gate,
                                   c->w.sel_pred_codebook, c->w.sel_succ_codebook, c->sel_tab, selected,
                                   nullptr, s, sel_smp);
       }));
  }
  return DFLASH_OK;
}

extern "C" dflash_status dflash_draft_step(dflash_ctx *c, void *stream, int32_t n_req,
                                           const int32_t *req_ids, const int32_t *anchors,
                                           int32_t *argmax, int32_t *topk_idx, float *topk_val,
                                           float *logits) {
  return draft_step_impl(c, stream, n_req, req_ids, anchors, argmax, topk_idx, topk_val, logits, nullptr);
}

extern "C" dflash_status dflash_draft_step_lse(dflash_ctx *c, void *stream, int32_t n_req,
                                               const int32_t *req_ids, const int32_t *anchors,
                                               int32_t *argmax, int32_t *topk_idx, float *topk_val,
                                               float *logits, float *lse) {
  return draft_step_impl(c, stream, n_req, req_ids, anchors, argmax, topk_idx, topk_val, logits, lse);
}

extern "C" dflash_status dflash_draft_step_ex(dflash_ctx *c, void *stream, int32_t n_req,
                                              const int32_t *req_ids, const int32_t *anchors,
                                              const dflash_draft_out *out) {
  if (!c) return DFLASH_ERR_INVALID_ARG;
  if (!out) return set_err(c, DFLASH_ERR_INVALID_ARG, "NULL outputs");
  SelSample smp{out->sel_temperature, out->sel_uniform, out->sel_q_tok, out->sel_q_p, out->sel_q_n};
  if (out->sel_uniform) {
    if (!out->selected || !out->sel_q_tok || !out->sel_q_p || !out->sel_q_n || !(out->sel_temperature > 0.f))
      return set_err(c, DFLASH_ERR_INVALID_ARG,
                     "the sampling walk needs selected, sel_q_tok/p/n and sel_temperature > 0");
  }
  return draft_step_impl(c, stream, n_req, req_ids, anchors, out->argmax, out->topk_idx, out->topk_val,
                         out->logits, out->lse, out->selected, out->sel_uniform ? &smp : nullptr);
}


// ------------------------------------------------------------------------------ verify / export
extern "C" dflash_status dflash_verify_greedy(dflash_ctx *c, void *stream, int32_t n_req,
                                              const int32_t *draft, const int32_t *target,
                                              int32_t *accept_len, int32_t *out_tokens,
                                              int32_t *next_anchor) {
  if (!c) return DFLASH_ERR_INVALID_ARG;
  dflash_status st = check_device_flag(c);
  if (st != DFLASH_OK) return st;
  if (n_req < 0) return set_err(c, DFLASH_ERR_INVALID_ARG, "n_req < 0");
  if (n_req == 0) return DFLASH_OK;
  if (!draft || !target || !accept_len || !out_tokens || !next_anchor)
    return set_err(c, DFLASH_ERR_INVALID_ARG, "NULL argument");
  DeviceGuard guard(c->device);
  if (guard.err != cudaSuccess) return set_err(c, DFLASH_ERR_CUDA, "cudaSetDevice failed");
  CK(c, timed(c, K_VERIFY, (cudaStream_t)stream, 4.0 * n_req * (3 * c->m.K + 4), (double)n_req * c->m.K, 1,
              [&] {
                return launch_verify(n_req, c->m.K, draft, target, accept_len, out_tokens,
                                     next_anchor, (cudaStream_t)stream);
              }));
  return DFLASH_OK;
}

static dflash_status check_sampling(dflash_ctx *c, const dflash_sampling *sp) {
  if (!sp) return set_err(c, DFLASH_ERR_INVALID_ARG, "NULL sampling parameters");
  if (sp->top_k == 0)
    return set_err(c, DFLASH_ERR_UNSUPPORTED, "top_k = 0 (top-p over the whole vocabulary) is not supported");
  if (!(sp->temperature > 0.f) || sp->top_k < 1 || sp->top_k > SMP_K || !(sp->top_p > 0.f) || sp->top_p > 1.f)
    return set_err(c, DFLASH_ERR_INVALID_ARG, "need temperature > 0, 1 <= top_k <= %d, 0 < top_p <= 1", SMP_K);
  return DFLASH_OK;
}

extern "C" dflash_status dflash_sample_tokens(dflash_ctx *c, void *stream, int32_t rows,
                                              const dflash_sampling *sp, const float *logits,
                                              const float *u, int32_t *tokens) {
  if (!c) return DFLASH_ERR_INVALID_ARG;
  dflash_status st = check_device_flag(c);
  if (st != DFLASH_OK) return st;
  if ((st = check_sampling(c, sp)) != DFLASH_OK) return st;
  if (rows < 0) return set_err(c, DFLASH_ERR_INVALID_ARG, "rows < 0");
  if (rows == 0) return DFLASH_OK;
  if (!logits || !u || !tokens) return set_err(c, DFLASH_ERR_INVALID_ARG, "NULL argument");
  DeviceGuard guard(c->device);
  if (guard.err != cudaSuccess) return set_err(c, DFLASH_ERR_CUDA, "cudaSetDevice failed");
  const int V = c->m.V;
  CK(c, timed(c, K_SAMPLE, (cudaStream_t)stream, 8.0 * rows * V, 4.0 * rows * V, 1, [&] {
       return launch_trunc_dist(rows, V, sp->temperature, sp->top_k, sp->top_p, logits, u, tokens,
                                nullptr, nullptr, nullptr, 2 * c->num_sms, (cudaStream_t)stream);
     }));
  return DFLASH_OK;
}

extern "C" dflash_status dflash_verify_sample(dflash_ctx *c, void *stream, int32_t n_req,
                                              const dflash_sampling *sp, const float *target_logits,
                                              const float *draft_logits, const int32_t *draft,
                                              const float *u_accept, const float *u_resample,
                                              int32_t *accept_len, int32_t *out_tokens,
                                              int32_t *next_anchor) {
  if (!c) return DFLASH_ERR_INVALID_ARG;
  dflash_status st = check_device_flag(c);
  if (st != DFLASH_OK) return st;
  if ((st = check_sampling(c, sp)) != DFLASH_OK) return st;
  if (n_req < 0 || n_req > c->cfg.max_batch)
    return set_err(c, DFLASH_ERR_INVALID_ARG, "n_req=%d outside [0, max_batch=%d]", n_req, c->cfg.max_batch);
  if (n_req == 0) return DFLASH_OK;
  if (!target_logits || !draft_logits || !draft || !u_accept || !u_resample || !accept_len || !out_tokens ||
      !next_anchor)
    return set_err(c, DFLASH_ERR_INVALID_ARG, "NULL argument");
  DeviceGuard guard(c->device);
  if (guard.err != cudaSuccess) return set_err(c, DFLASH_ERR_CUDA, "cudaSetDevice failed");
  cudaStream_t s = (cudaStream_t)stream;
  const int V = c->m.V, K = c->m.K, Q = c->m.Q();
  const int tr = n_req * Q, dr = n_req * K;
  int32_t *ptok = c->smp_tok, *qtok = c->smp_tok + (size_t)tr * SMP_K;
  float *pp = c->smp_p, *qp = c->smp_p + (size_t)tr * SMP_K;
  int32_t *pn = c->smp_n, *qn = c->smp_n + tr;
  CK(c, timed(c, K_SAMPLE, s, 4.0 * (tr + dr) * V, 4.0 * (tr + dr) * V, 2, [&] {
       cudaError_t e = launch_trunc_dist(tr, V, sp->temperature, sp->top_k, sp->top_p, target_logits,
                                         nullptr, nullptr, ptok, pp, pn, 2 * c->num_sms, s);
       if (e != cudaSuccess) return e;
       return launch_trunc_dist(dr, V, sp->temperature, sp->top_k, sp->top_p, draft_logits, nullptr,
                                nullptr, qtok, qp, qn, 2 * c->num_sms, s);
     }));
  CK(c, timed(c, K_VERIFY, s, 4.0 * n_req * (3 * K + 4), (double)n_req * K, 1, [&] {
       return launch_verify_sample(n_req, K, ptok, pp, pn, qtok, qp, qn, draft, u_accept, u_resample,
                                   accept_len, out_tokens, next_anchor, s);
     }));
  return DFLASH_OK;
}

extern "C" dflash_status dflash_verify_sample_q(dflash_ctx *c, void *stream, int32_t n_req,
                                                const dflash_sampling *sp, const float *target_logits,
                                                const int32_t *q_tok, const float *q_p, const int32_t *q_n,
                                                const int32_t *draft, const float *u_accept,
                                                const float *u_resample, int32_t *accept_len,
                                                int32_t *out_tokens, int32_t *next_anchor) {
  if (!c) return DFLASH_ERR_INVALID_ARG;
  dflash_status st = check_device_flag(c);
  if (st != DFLASH_OK) return st;
  if ((st = check_sampling(c, sp)) != DFLASH_OK) return st;
  if (n_req < 0 || n_req > c->cfg.max_batch)
    return set_err(c, DFLASH_ERR_INVALID_ARG, "n_req=%d outside [0, max_batch=%d]", n_req, c->cfg.max_batch);
  if (n_req == 0) return DFLASH_OK;
  if (!target_logits || !q_tok || !q_p || !q_n || !draft || !u_accept || !u_resample || !accept_len ||
      !out_tokens || !next_anchor)
    return set_err(c, DFLASH_ERR_INVALID_ARG, "NULL argument");
  DeviceGuard guard(c->device);
  if (guard.err != cudaSuccess) return set_err(c, DFLASH_ERR_CUDA, "cudaSetDevice failed");
  cudaStream_t s = (cudaStream_t)stream;
  const int V = c->m.V, K = c->m.K, Q = c->m.Q();
  const int tr = n_req * Q;
  CK(c, timed(c, K_SAMPLE, s, 4.0 * tr * V, 4.0 * tr * V, 1, [&] {
       return launch_trunc_dist(tr, V, sp->temperature, sp->top_k, sp->top_p, target_logits, nullptr, nullptr,
                                c->smp_tok, c->smp_p, c->smp_n, 2 * c->num_sms, s);
     }));
  CK(c, timed(c, K_VERIFY, s, 4.0 * n_req * (3 * K + 4), (double)n_req * K, 1, [&] {
       return launch_verify_sample(n_req, K, c->smp_tok, c->smp_p, c->smp_n, q_tok, q_p, q_n, draft, u_accept,
                                   u_resample, accept_len, out_tokens, next_anchor, s);
     }));
  return DFLASH_OK;
}

extern "C" dflash_status dflash_export_kv(dflash_ctx *c, void *stream, int32_t req_id, int32_t layer,
                                          int32_t pos0, int32_t n, void *k_out, void *v_out) {
  if (!c) return DFLASH_ERR_INVALID_ARG;
  dflash_status st = check_device_flag(c);
  if (st != DFLASH_OK) return st;
  auto it = c->reqs.find(req_id);
  if (it == c->reqs.end()) return set_err(c, DFLASH_ERR_UNKNOWN_REQUEST, "unknown request %d", req_id);
  const Req &q = it->second;
  if (layer < 0 || layer >= c->m.L || pos0 < 0 || n < 0 || pos0 + n > q.len)
    return set_err(c, DFLASH_ERR_INVALID_ARG, "export range outside the context");
  if (n == 0) return DFLASH_OK;
  if (!k_out || !v_out) return set_err(c, DFLASH_ERR_INVALID_ARG, "NULL output");
  DeviceGuard guard(c->device);
  if (guard.err != cudaSuccess) return set_err(c, DFLASH_ERR_CUDA, "cudaSetDevice failed");
  cudaStream_t s = (cudaStream_t)stream;
  const int32_t *dp = nullptr;
  if ((st = stage_upload(c, s, q.pages.data(), q.pages.size() * 4, &dp)) != DFLASH_OK) return st;
  CK(c, timed(c, K_EXPORT, s, 4.0 * n * c->m.kv_dim() * c->esz, 0.0, 1, [&] {
       return launch_export_kv(c->dtype, c->m, layer, pos0, n, dp, c->pool, k_out, v_out, s);
     }));
  return DFLASH_OK;
}

// ------------------------------------------------------------------------------ timing
extern "C" dflash_status dflash_timing_enable(dflash_ctx *c, int32_t enable) {
  if (!c) return DFLASH_ERR_INVALID_ARG;
  c->timing = enable != 0;
  return DFLASH_OK;
}

extern "C" int32_t dflash_timing_classes(void) { return K_NUM; }

extern "C" const char *dflash_timing_class_name(int32_t cls) {
  return (cls >= 0 && cls < K_NUM) ? kClsName[cls] : "";
}

extern "C" dflash_status dflash_timing_read(dflash_ctx *c, double *ms, int64_t *launches,
                                            double *bytes, double *flops, int32_t n) {
  if (!c || n < 0) return DFLASH_ERR_INVALID_ARG;
  DeviceGuard guard(c->device);
  dflash_status st = DFLASH_OK;
  for (const TimeRec &r : c->recs) {
    float t = 0.f;
    cudaError_t e = cudaEventSynchronize(r.b);
    if (e == cudaSuccess) e = cudaEventElapsedTime(&t, r.a, r.b);
    if (e != cudaSuccess && st == DFLASH_OK)
      st = set_err(c, DFLASH_ERR_CUDA, "timing event: %s", cudaGetErrorString(e));
    if (r.cls < n) {
      if (ms) ms[r.cls] += t;
      if (launches) launches[r.cls] += r.launches;
      if (bytes) bytes[r.cls] += r.bytes;
      if (flops) flops[r.cls] += r.flops;
    }
    c->spare_events.push_back(r.a);
    c->spare_events.push_back(r.b);
  }
  c->recs.clear();
  return st;
}
