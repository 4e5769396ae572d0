// C ABI of the frame decoder: context, workspace layout, phase programs, call drivers.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "s2_internal.h"

using namespace s2;

struct s2_ctx {
  Dims d{};
  const void *E = nullptr, *CE = nullptr, *norm = nullptr, *P = nullptr, *FE = nullptr, *fnorm = nullptr,
             *FO = nullptr;
  std::vector<LayerW> slow, fast;
  unsigned char* ws = nullptr;
  size_t ws_bytes = 0;
  int max_streams = 0, kv_slots = 0, grid = 0, device = 0;
  // workspace regions
  Control* ctl = nullptr;
  float2* rope = nullptr;
  float2* rope_f = nullptr;
  StreamState* st = nullptr;       // [max_streams + 1] (last: scratch state of the Fast-AR-alone path)
  float* hidden = nullptr;         // [max_streams + 1][D]
  float* logits = nullptr;         // [max_streams][A]
  unsigned char* kc = nullptr;     // [L][max_streams][Hkv][slots][hd]
  unsigned char* vc = nullptr;
  int32_t* stage = nullptr;        // [max_streams][kMaxFramesPerCall][NCB]
  float *x = nullptr, *qkv = nullptr, *o = nullptr, *g = nullptr;
  float *fx = nullptr, *fqkv = nullptr, *fo = nullptr, *fg = nullptr, *fk = nullptr, *fv = nullptr;
  // bf16 hi / lo rows of projection inputs (bf16 models): attention outputs and SwiGLU outputs
  uint16_t *op = nullptr, *gp = nullptr, *fop = nullptr, *fgp = nullptr;
  float *flogits = nullptr, *part = nullptr, *pscratch = nullptr;
  int32_t* fcode = nullptr;
  Phase* prog = nullptr;           // [max_streams][n_dec] then fast-only program
  int n_dec = 0, n_fast = 0, prefill_chunk = 0;
  unsigned long long* trace = nullptr;  // caller-owned device buffer (tracing hook)
  int trace_cap = 0;
  unsigned gbar_base = 0;          // grid-barrier counter start (test hook)
  unsigned tag_next = 1;           // tag counter of the tagged handoffs (per launch: take_tags)
  std::vector<int> host_pos;
  std::vector<char> host_prefilled;
  std::string err;
  // batched decode (bf16 models serving several streams)
  bool batched = false;
  int sms = 0;
  BatchModel bm{};
  Batch* batch = nullptr;
  uint16_t* pf_planes = nullptr;   // prompt projections: planes [256][pf_ld]
  int pf_ld = 0;
  float* pf_part = nullptr;
  std::vector<QuantW> qw;          // fp8 weight streaming: e4m3 copies of the projections
  int* qbad = nullptr;             // expansion check result
};

namespace {

std::string g_init_error = "no error";

constexpr const char* kLayerNames[9] = {"attention_norm", "attention.wqkv", "attention.q_norm", "attention.k_norm",
                                        "attention.wo", "ffn_norm", "feed_forward.w1", "feed_forward.w3",
                                        "feed_forward.w2"};

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
// floats between the admissible-logit rows of consecutive streams: rows start on 256-byte
// boundaries (the sampler copies a row into shared memory in 16-byte pieces)
size_t logits_stride(const Dims& d) { return align_up(static_cast<size_t>(d.A), 64); }

// Every activation-plane pointer of a program lies, with its whole extent, inside
// [base, base + bytes): the device reads and writes them without further checks.
bool planes_inside(const Phase* prog, size_t n, const void* base, size_t bytes, std::string& why) {
  const uintptr_t lo = reinterpret_cast<uintptr_t>(base), hi = lo + bytes;
  auto in = [&](const void* q, size_t m) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(q);
    return a >= lo && a + m <= hi;
  };
  for (size_t i = 0; i < n; ++i) {
    const Phase& p = prog[i];
    if (p.op == OP_GEMV) {
      for (int c = 0; c < p.ncols; ++c) {
        const size_t in_b = (p.col[c].tag_back > 0 ? 8ull : 4ull) * p.K, out_b = (p.tag_out ? 8ull : 4ull) * p.M;
        if (p.col[c].src == SRC_PLANES && !in(p.col[c].p, in_b)) return (why = "planes input outside the workspace", false);
        if (p.yp[c] != nullptr && !in(p.yp[c], out_b)) return (why = "planes output outside the workspace", false);
      }
    }
    if ((p.op == OP_ATTN_SLOW || p.op == OP_ATTN_FAST) && p.outp != nullptr &&
        !in(p.outp, 4ull * static_cast<size_t>(p.npos > 0 ? p.npos : 1)))
      return (why = "attention planes outside the workspace", false);
  }
  return true;
}

int fail(s2_ctx* c, int code, const std::string& msg) {
  if (c) c->err = msg;
  else g_init_error = msg;
  return code;
}

bool to_dims(const s2_dims* s, Dims& d, std::string& why) {
  d.D = s->dim; d.L = s->n_layer; d.Hq = s->n_head; d.Hkv = s->n_kv_head; d.hd = s->head_dim; d.F = s->ffn;
  d.V = s->vocab; d.sem_lo = s->sem_begin; d.sem_hi = s->sem_end; d.im_end = s->im_end; d.ncb = s->n_codebooks;
  d.cbs = s->codebook_size; d.sem_scale = s->sem_scale; d.eps = s->norm_eps; d.rope_base = s->rope_base;
  d.qk_norm = s->qk_norm; d.rope_bf16 = s->rope_table_bf16; d.Df = s->fast_dim; d.Lf = s->fast_n_layer;
  d.Hqf = s->fast_n_head; d.Hkvf = s->fast_n_kv_head; d.hdf = s->fast_head_dim; d.Ff = s->fast_ffn;
  d.Wf = s->fast_window; d.has_proj = s->has_fast_project_in; d.wdt = s->weight_dtype; d.kvdt = s->kv_dtype;
  d.fp8 = s->weight_fp8;
  d.esz = d.wdt == S2_BF16 ? 2 : 4;
  d.kvsz = d.kvdt == S2_F16 ? 2 : 4;
  d.A = d.cbs + 1;
  auto bad = [&](const char* m) { why = m; return false; };
  if (d.wdt != S2_BF16 && d.wdt != S2_F32) return bad("weight_dtype must be S2_BF16 or S2_F32");
  if (d.kvdt != S2_F16 && d.kvdt != S2_F32) return bad("kv_dtype must be S2_F16 or S2_F32");
  if ((d.wdt == S2_BF16) != (d.kvdt == S2_F16)) return bad("bf16 weights go with an S2_F16 KV cache, fp32 weights with S2_F32");
  if (d.fp8 != 0 && d.fp8 != 1) return bad("weight_fp8 must be 0 or 1");
  if (d.fp8 && d.wdt != S2_BF16) return bad("fp8 weight streaming needs bf16 weights");
  if (d.fp8 && (d.D % 128 || d.Df % 128 || d.F % 128 || d.Ff % 128 || (d.Hq * d.hd) % 128 || (d.Hqf * d.hdf) % 128))
    return bad("fp8 weight streaming needs projection lengths that are multiples of 128");
  const int al = d.wdt == S2_BF16 ? 8 : 4;
  if (d.D <= 0 || d.D % al || d.Df <= 0 || d.Df % al) return bad("dim/fast_dim must be positive multiples of 16 bytes");
  if (d.L < 0 || d.Lf <= 0) return bad("a fast decoder (fast_n_layer > 0) is required");
  if (d.ncb < 2 || d.ncb > kMaxCodebooks) return bad("n_codebooks out of range (2..15)");
  if (d.Wf < d.ncb || d.Wf > 16) return bad("fast_window must cover n_codebooks positions (and be <= 16)");
  if (d.cbs <= 0 || d.cbs % al) return bad("codebook_size must be a positive multiple of 16 bytes of weights");
  if (d.Hqf <= 0 || d.Hkvf <= 0 || d.Hqf % d.Hkvf || d.Hqf / d.Hkvf > 4) return bad("fast heads: n_head % n_kv_head == 0, ratio <= 4");
  if (d.hdf != 64 && d.hdf != 128) return bad("fast_head_dim must be 64 or 128");
  if (d.Ff <= 0 || d.Ff % al || (d.Hqf * d.hdf) % al) return bad("fast ffn / head sizes must be multiples of 16 bytes");
  if (!d.has_proj && d.Df != d.D) return bad("without fast_project_in, fast_dim must equal dim");
  if (!(d.sem_scale > 0.f) || !(d.eps > 0.f) || !(d.rope_base > 1.0)) return bad("sem_scale, norm_eps, rope_base must be positive");
  if (d.qk_norm != 0 && d.qk_norm != 1) return bad("qk_norm must be 0 or 1");
  if (d.L > 0) {
    if (d.Hq <= 0 || d.Hkv <= 0 || d.Hq % d.Hkv || d.Hq / d.Hkv > 4 || d.Hkv > 64) return bad("heads: n_head % n_kv_head == 0, ratio <= 4, n_kv_head <= 64");
    if (d.hd != 64 && d.hd != 128) return bad("head_dim must be 64 or 128");
    if (d.hd != d.hdf) return bad("head_dim and fast_head_dim must be equal");
    if (d.F <= 0 || d.F % al || (d.Hq * d.hd) % al) return bad("ffn / head sizes must be multiples of 16 bytes");
    if (d.sem_hi - d.sem_lo + 1 != d.cbs) return bad("the semantic range must hold codebook_size ids");
    if (d.sem_lo < 0 || d.sem_hi >= d.V || d.im_end < 0 || d.im_end >= d.V) return bad("semantic range / im_end outside the vocabulary");
    if (d.im_end >= d.sem_lo && d.im_end <= d.sem_hi) return bad("im_end must lie outside the semantic range");
  }
  const int64_t maxk = kStageBytes / d.esz;
  if (d.D > maxk || d.F > maxk || d.Ff > maxk || d.Hq * d.hd > maxk || d.Hqf * d.hdf > maxk || d.Df > maxk)
    return bad("a projection input is longer than one pipeline stage");
  if (2LL * d.D * d.esz > kStageBytes || 2LL * d.Df * d.esz > kStageBytes) return bad("gate/up rows exceed one pipeline stage");
  return true;
}

int layer_count(const Dims& d) { return 3 + 9 * d.L + 4 + 9 * d.Lf; }

long long tensor_numel(const Dims& d, int i, std::string* name) {
  auto setn = [&](const std::string& s) { if (name) *name = s; };
  if (i < 0 || i >= layer_count(d)) return -1;
  if (i == 0) { setn("embeddings"); return 1LL * d.V * d.D; }
  if (i == 1) { setn("codebook_embeddings"); return 1LL * d.ncb * d.cbs * d.D; }
  if (i == 2) { setn("norm"); return d.D; }
  i -= 3;
  auto layer = [&](int li, int k, const char* pre, int D, int Hq, int Hkv, int hd, int F) -> long long {
    setn(std::string(pre) + std::to_string(li) + "." + kLayerNames[k]);
    switch (k) {
      case 0: case 5: return D;
      case 1: return 1LL * (Hq + 2 * Hkv) * hd * D;
      case 2: case 3: return hd;
      case 4: return 1LL * D * Hq * hd;
      case 6: case 7: return 1LL * F * D;
      default: return 1LL * D * F;
    }
  };
  if (i < 9 * d.L) return layer(i / 9, i % 9, "layers.", d.D, d.Hq, d.Hkv, d.hd, d.F);
  i -= 9 * d.L;
  if (i == 0) { setn("fast_project_in"); return 1LL * d.Df * d.D; }
  if (i == 1) { setn("fast_embeddings"); return 1LL * d.cbs * d.Df; }
  if (i == 2) { setn("fast_norm"); return d.Df; }
  if (i == 3) { setn("fast_output"); return 1LL * d.cbs * d.Df; }
  i -= 4;
  return layer(i / 9, i % 9, "fast_layers.", d.Df, d.Hqf, d.Hkvf, d.hdf, d.Ff);
}

// Sequential carve of the workspace (base == nullptr: size only).
struct Carver {
  unsigned char* base;
  size_t off = 0;
  template <typename T>
  T* take(size_t count) {
    off = align_up(off, 256);
    T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
    off += count * sizeof(T);
    return p;
  }
};

// A 2-column bf16 projection stages 2 x 2 padded rows of K bf16 activations in shared memory; the Fast-AR
// down projection of the first call (two positions) is split when that does not fit.
bool split_fast_down(const Dims& d, int npos) {
  return npos == 2 && d.wdt == S2_BF16 && 2LL * 2 * (2LL * d.Ff + kTileRowPad) > kXsBytes;
}

int fast_call_phases(const Dims& d) {
  int n = 0;
  for (int cb = 1; cb < d.ncb; ++cb) n += d.Lf * (5 + (split_fast_down(d, cb == 1 ? 2 : 1) ? 1 : 0)) + 2;
  return n;
}

int fast_alone_phases(const Dims& d) { return 2 + fast_call_phases(d); }

int attn_items_max(const Dims& d, int grid, int slots) {
  if (d.L == 0) return 1;
  return d.Hkv * (grid / d.Hkv + slots / kAttnMaxChunk + 2);
}

// bf16 contexts serving several streams also carry the batched-decode buffers
void setup_batched(s2_ctx* c) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      sms <= 0) {
    cudaGetLastError();
    sms = 152;
  }
  c->sms = sms;
  c->batched = batch_supported(c->d, c->max_streams, nullptr);
}

void carve(s2_ctx* c, Carver& cv) {
  const Dims& d = c->d;
  const int B = c->max_streams;
  const size_t slots = static_cast<size_t>(c->kv_slots);
  const int QKV = (d.Hq + 2 * d.Hkv) * d.hd, QKVf = (d.Hqf + 2 * d.Hkvf) * d.hdf;
  c->ctl = cv.take<Control>(1);
  c->rope = cv.take<float2>(std::max<size_t>(1, slots * (d.hd / 2)));
  c->rope_f = cv.take<float2>(static_cast<size_t>(d.Wf) * (d.hdf / 2));
  c->st = cv.take<StreamState>(B + 1);
  c->hidden = cv.take<float>(static_cast<size_t>(B + 1) * d.D);
  c->logits = cv.take<float>(static_cast<size_t>(B) * logits_stride(d));
  const size_t kv = static_cast<size_t>(d.L) * B * d.Hkv * slots * d.hd * d.kvsz;
  c->kc = cv.take<unsigned char>(kv);
  c->vc = cv.take<unsigned char>(kv);
  c->stage = cv.take<int32_t>(static_cast<size_t>(B) * kMaxFramesPerCall * d.ncb);
  c->x = cv.take<float>(2 * static_cast<size_t>(d.D));  // tagged words (bf16 models)
  c->qkv = cv.take<float>(2 * static_cast<size_t>(std::max(QKV, 1)));  // tagged words (bf16 models)
  c->o = cv.take<float>(std::max(d.Hq * d.hd, 1));
  c->g = cv.take<float>(std::max(d.F, 1));
  c->fx = cv.take<float>(2 * static_cast<size_t>(d.Wf) * d.Df);
  c->fqkv = cv.take<float>(4 * static_cast<size_t>(QKVf));  // two positions of tagged words
  c->fo = cv.take<float>(2 * static_cast<size_t>(d.Hqf) * d.hdf);
  c->fg = cv.take<float>(2 * static_cast<size_t>(d.Ff));
  c->op = cv.take<uint16_t>(2 * static_cast<size_t>(std::max(d.Hq * d.hd, 1)));
  c->gp = cv.take<uint16_t>(4 * static_cast<size_t>(std::max(d.F, 1)));
  c->fop = cv.take<uint16_t>(4 * static_cast<size_t>(d.Hqf) * d.hdf);
  c->fgp = cv.take<uint16_t>(8 * static_cast<size_t>(d.Ff));
  c->fk = cv.take<float>(static_cast<size_t>(d.Lf) * d.Wf * d.Hkvf * d.hdf);
  c->fv = cv.take<float>(static_cast<size_t>(d.Lf) * d.Wf * d.Hkvf * d.hdf);
  c->flogits = cv.take<float>(d.cbs);
  c->fcode = cv.take<int32_t>(16);
  c->part = cv.take<float>(static_cast<size_t>(attn_items_max(d, c->grid, c->kv_slots)) * 4 * (d.hd + 2));
  c->prefill_chunk = 512;
  c->pscratch = d.L > 0 ? cv.take<float>(prefill_scratch_floats(d, c->prefill_chunk)) : nullptr;
  c->n_dec = d.L > 0 ? 1 + fast_call_phases(d) + 5 * d.L + 1 : 0;
  c->n_fast = fast_alone_phases(d);
  c->prog = cv.take<Phase>(static_cast<size_t>(B) * c->n_dec + c->n_fast);
  if (c->batched) {
    const BatchSizes z = batch_sizes(d, B, c->sms);
    BatchModel& m = c->bm;
    m.pX = cv.take<uint16_t>(z.planes_rows * z.ldX);
    m.pO = cv.take<uint16_t>(z.planes_rows * z.ldO);
    m.pH = cv.take<uint16_t>(z.planes_rows * z.ldH);
    m.part = cv.take<float>(z.part_floats);
    m.bx = cv.take<float>(static_cast<size_t>(B) * d.D);
    m.bfx = cv.take<float>(static_cast<size_t>(B) * 2 * d.Df);
    const size_t fw = static_cast<size_t>(B) * d.Lf * d.Wf * d.Hkvf * d.hdf;
    m.bfk = cv.take<float>(fw);
    m.bfv = cv.take<float>(fw);
    m.apart = cv.take<float>(z.apart_floats);
    m.bflog = cv.take<float>(static_cast<size_t>(B) * d.cbs);
    m.bfcode = cv.take<int32_t>(static_cast<size_t>(B) * 16);
    m.bctl = cv.take<int>(16);
    m.bstreams = cv.take<unsigned char>(batch_stream_bytes(B));
    // prompt projections on the tensor cores: planes of up to 128 positions and their partials
    c->pf_ld = std::max(std::max(d.D, d.Hq * d.hd), d.F);
    c->pf_planes = cv.take<uint16_t>(static_cast<size_t>(2 * kPrefillChunkTC) * c->pf_ld);
    c->pf_part = cv.take<float>(batch_prefill_part_floats(d, c->sms));
  }
  // fp8 weight streaming: e4m3 codes + row scales of every projection matrix
  c->qw.clear();
  if (d.fp8) {
    auto addq = [&](const void* w, long long rows, int cols) {
      QuantW q{};
      q.w = w;
      q.rows = rows;
      q.cols = cols;
      q.q = cv.take<uint8_t>(static_cast<size_t>(rows) * cols);
      q.s = cv.take<float>(static_cast<size_t>(rows));
      c->qw.push_back(q);
    };
    auto layers = [&](const std::vector<LayerW>& v, int n, int D, int qkv, int hq, int F) {
      for (int l = 0; l < n; ++l) {
        const bool have = l < static_cast<int>(v.size());
        addq(have ? v[l].wqkv : nullptr, qkv, D);
        addq(have ? v[l].wo : nullptr, D, hq);
        addq(have ? v[l].w1 : nullptr, F, D);
        addq(have ? v[l].w3 : nullptr, F, D);
        addq(have ? v[l].w2 : nullptr, D, F);
      }
    };
    layers(c->slow, d.L, d.D, QKV, d.Hq * d.hd, d.F);
    layers(c->fast, d.Lf, d.Df, QKVf, d.Hqf * d.hdf, d.Ff);
    if (d.has_proj) addq(c->P, d.Df, d.D);
    addq(c->FO, d.cbs, d.Df);
    c->qbad = cv.take<int>(1);
  }
}

// ------------------------------------------------------------ phase builders

// Base tag of a launch of `count` phases from a running counter: tags are never 0 (the value the
// tagged buffers are cleared to), and a launch's tags do not wrap around 2^32.
unsigned take_tags(unsigned& ctr, long long count) {
  if (ctr == 0u || static_cast<unsigned long long>(ctr) + static_cast<unsigned long long>(count) + 1ull > 0xffffffffull)
    ctr = 1u;
  const unsigned t = ctr;
  ctr += static_cast<unsigned>(count) + 1u;
  return t;
}

// The buffers the Fast-AR phases read and write: a context's workspace regions or the static
// array's (s2_fast_logits_static).
struct FastBufs {
  float* hidden_src;  // the hidden feeding Fast-AR position 0
  float *fx, *fqkv, *fo, *fg, *fk, *fv, *flogits;
  uint16_t *fop, *fgp;  // bf16 hi / lo rows of the attention and SwiGLU outputs (bf16 models)
  int32_t* fcode;
};

// The Fast-AR weights (device pointers of the weight table)
struct FastWts {
  const LayerW* layers;  // [fast_n_layer]
  const void *P, *FO, *fnorm;
};

// Appends phases to a caller-given array (no allocation); `n` counts every push, so a program
// longer than `cap` is detected by the caller (n > cap) without writing past the array.
struct Builder {
  Dims d;
  int grid;
  Phase* out;
  int cap;
  int n = 0;
  std::string err;
  // tagged buffers (bf16 models: the residual rows and the SwiGLU planes) and the index of the
  // phase that last wrote each of them in the program being built
  std::vector<std::pair<const unsigned char*, size_t>> tagged_ranges;
  std::vector<std::pair<const void*, int>> last_write;

  bool tagged() const { return d.wdt == S2_BF16; }
  int xw() const { return tagged() ? 2 : 1; }  // floats per residual element
  int pw() const { return tagged() ? 4 : 2; }  // 16-bit units per planes element
  void add_tagged(const void* p, size_t bytes) {
    if (tagged()) tagged_ranges.emplace_back(static_cast<const unsigned char*>(p), bytes);
  }
  bool is_tagged(const void* p) const {
    const unsigned char* q = static_cast<const unsigned char*>(p);
    for (const auto& r : tagged_ranges)
      if (q >= r.first && q < r.first + r.second) return true;
    return false;
  }
  void new_program() { last_write.clear(); }
  int* lw(const void* p) {
    for (auto& e : last_write)
      if (e.first == p) return &e.second;
    return nullptr;
  }
  void wrote(const void* p) {
    if (int* w = lw(p)) *w = n;
    else last_write.emplace_back(p, n);
  }
  // tagged inputs take the distance to their writer; tagged outputs and write-backs are recorded;
  // the residual-add and SwiGLU projections, and a projection whose output only the next
  // (attention) phase reads (`polled`), hand over without a grid barrier
  void tag(Phase& p, bool polled) {
    if (!tagged()) return;
    if (p.op == OP_ATTN_SLOW || p.op == OP_ATTN_FAST) {
      if (is_tagged(p.qkv)) {
        const int* w = lw(p.qkv);
        if (!w) err = "internal: a tagged attention input is read before it is written";
        else p.qkv_tag_back = n - *w;
      }
      return;
    }
    if (p.op != OP_GEMV) return;
    for (int c = 0; c < p.ncols; ++c) {
      const GemvCol& col = p.col[c];
      if ((col.src == SRC_BUF || col.src == SRC_PLANES) && is_tagged(col.p)) {
        const int* w = lw(col.p);
        if (!w) {
          err = "internal: a tagged input is read before it is written";
          continue;
        }
        p.col[c].tag_back = n - *w;
      }
    }
    bool any_t = false, any_u = false;
    for (int c = 0; c < p.ncols; ++c) {
      for (const void* o : {static_cast<const void*>(p.y[c]), static_cast<const void*>(p.yp[c])}) {
        if (!o) continue;
        (is_tagged(o) ? any_t : any_u) = true;
      }
    }
    if (any_t && any_u) err = "internal: a phase mixes tagged and plain outputs";
    p.tag_out = any_t ? 1 : 0;
    p.no_sync = (any_t && (p.epi == EPI_ADD || p.epi == EPI_SWIGLU || polled)) ? 1 : 0;
    for (int c = 0; c < p.ncols; ++c) {
      if (p.y[c] && any_t) wrote(p.y[c]);
      if (p.yp[c] && any_t) wrote(p.yp[c]);
      if (p.col[c].wb) {
        if (!is_tagged(p.col[c].wb)) err = "internal: a column write-back outside the tagged buffers";
        wrote(p.col[c].wb);
      }
    }
  }

  Phase gemv(int M, int K, int ncols, const void* w0, const void* w1, const void* normw, int epi) {
    Phase p{};
    p.op = OP_GEMV;
    p.M = M;
    p.K = K;
    p.nmat = w1 ? 2 : 1;
    p.ncols = ncols;
    p.epi = epi;
    p.w[0] = w0;
    p.w[1] = w1;
    p.normw = normw;
    const int epc = 16 / d.esz;
    const int nchunk = K / epc;
    // every consumer warp takes a 1/8 K-slice of every row (all warps on every tile)
    const int Q = kConsumerWarps;
    if ((nchunk + Q - 1) / Q > 32 * kGemvChunksPerLane) err = "projection too long for the register-resident activation slices";
    p.Q = Q;
    const int rowb = K * d.esz * p.nmat;
    p.rows_per_tile = std::max(1, kStageBytes / rowb);
    if (d.wdt == S2_BF16) {
      // 8-row tiles of Kt columns: Kt a multiple of 16 dividing K, 8 padded rows within a stage
      const int kmax = (kStageBytes / kTileRows - kTileRowPad) / 2;
      int nkt = (K + kmax - 1) / kmax;
      while (nkt <= K / 16 && (K % nkt != 0 || (K / nkt) % 16 != 0)) ++nkt;
      if (nkt > K / 16) err = "no K tiling of a projection fits the pipeline stage";
      p.Kt = K / nkt;
      p.nkt = nkt;
      if (2LL * ncols * (2LL * K + kTileRowPad) > kXsBytes) err = "projection input does not fit the shared activation buffer";
      if (K * d.esz > kStageBytes) err = "norm vector exceeds one pipeline stage";
    }
    return p;
  }
  void push(Phase p, bool polled = false) {
    tag(p, polled);
    const int g2 = grid - p.cta0;
    if (g2 > 0) {
      // the device splits the rows without dividing (rows_of)
      p.rows_base = p.M / g2;
      p.rows_rem = p.M % g2;
    }
    if (p.op == OP_GEMV && p.ncols == 2 && (p.col[0].src == SRC_PLANES) != (p.col[1].src == SRC_PLANES))
      err = "internal: a phase mixes planes and other activation sources";
    if (p.op == OP_GEMV && p.col[0].src == SRC_PLANES && p.normw != nullptr) err = "internal: normalised planes input";
    if (p.op == OP_GEMV) {
      const int rows = (p.M + g2 - 1) / g2;
      if (static_cast<long long>(rows) * p.nmat * p.ncols * kConsumerWarps > kRedFloats)
        err = "too many rows per CTA for the partial-sum buffer";
      if (p.last_row && p.nmat != 1) err = "last-row override needs one matrix";
    }
    if (n < cap) out[n] = p;
    ++n;
  }
  static GemvCol buf(const float* p, float* wb = nullptr) { return GemvCol{SRC_BUF, 0, p, wb}; }
  static GemvCol planes(const uint16_t* p) { return GemvCol{SRC_PLANES, 0, p, nullptr}; }
  // bf16 models pass attention and SwiGLU outputs to the next projection as hi / lo planes
  bool use_planes() const { return d.wdt == S2_BF16; }

  // Fast-AR calls 1..NCB-1, each followed by its draw (ch.06 §1-§4): positions 0 and 1 in the
  // first call, then one new position per call over the within-frame K/V
  void fast_calls(const FastBufs& b, const FastWts& w) {
    const int QKVf = (d.Hqf + 2 * d.Hkvf) * d.hdf;
    const size_t kvl = static_cast<size_t>(d.Wf) * d.Hkvf * d.hdf;
    const float scale = static_cast<float>(1.0 / std::sqrt(static_cast<double>(d.hdf)));
    for (int cb = 1; cb < d.ncb; ++cb) {
      const int npos = cb == 1 ? 2 : 1, pos0 = cb == 1 ? 0 : cb;
      for (int l = 0; l < d.Lf; ++l) {
        const LayerW& lw = w.layers[l];
        Phase q = gemv(QKVf, d.Df, npos, lw.wqkv, nullptr, lw.an, EPI_STORE);
        for (int j = 0; j < npos; ++j) {
          const int p = pos0 + j;
          float* xp = b.fx + static_cast<size_t>(p) * d.Df * xw();
          if (l == 0 && p >= 1) q.col[j] = GemvCol{SRC_FEROW, 0, b.fcode + (p - 1), xp};
          else if (l == 0 && p == 0 && !d.has_proj) q.col[j] = buf(b.hidden_src, xp);
          else q.col[j] = buf(xp);
          q.y[j] = b.fqkv + static_cast<size_t>(j) * QKVf * xw();
        }
        push(q, true);  // read only by the attention phase that follows, which polls its words
        Phase a{};
        a.op = OP_ATTN_FAST;
        a.layer = l;
        a.npos = npos;
        a.pos0 = pos0;
        a.qkv = b.fqkv;
        a.out = b.fo;
        if (use_planes()) a.outp = b.fop;
        a.kc = b.fk + l * kvl;
        a.vc = b.fv + l * kvl;
        a.qn = lw.qn;
        a.kn = lw.kn;
        a.scale = scale;
        push(a);
        Phase o = gemv(d.Df, d.Hqf * d.hdf, npos, lw.wo, nullptr, nullptr, EPI_ADD);
        for (int j = 0; j < npos; ++j) {
          o.col[j] = use_planes() ? planes(b.fop + static_cast<size_t>(j) * 2 * d.Hqf * d.hdf)
                                  : buf(b.fo + static_cast<size_t>(j) * d.Hqf * d.hdf);
          o.y[j] = b.fx + static_cast<size_t>(pos0 + j) * d.Df * xw();
        }
        push(o);
        Phase u = gemv(d.Ff, d.Df, npos, lw.w1, lw.w3, lw.fn, EPI_SWIGLU);
        for (int j = 0; j < npos; ++j) {
          u.col[j] = buf(b.fx + static_cast<size_t>(pos0 + j) * d.Df * xw());
          if (use_planes()) u.yp[j] = b.fgp + static_cast<size_t>(j) * d.Ff * pw();
          else u.y[j] = b.fg + static_cast<size_t>(j) * d.Ff;
        }
        push(u);
        // two positions whose activations exceed the shared buffer: one down phase per position
        const int ndown = split_fast_down(d, npos) ? npos : 1;
        for (int t = 0; t < ndown; ++t) {
          const int nc = ndown == 1 ? npos : 1;
          Phase dn = gemv(d.Df, d.Ff, nc, lw.w2, nullptr, nullptr, EPI_ADD);
          for (int j = 0; j < nc; ++j) {
            const int jj = ndown == 1 ? j : t;
            dn.col[j] = use_planes() ? planes(b.fgp + static_cast<size_t>(jj) * d.Ff * pw())
                                     : buf(b.fg + static_cast<size_t>(jj) * d.Ff);
            dn.y[j] = b.fx + static_cast<size_t>(pos0 + jj) * d.Df * xw();
          }
          push(dn);
        }
      }
      Phase fo = gemv(d.cbs, d.Df, 1, w.FO, nullptr, w.fnorm, EPI_STORE);
      fo.col[0] = buf(b.fx + static_cast<size_t>(cb) * d.Df * xw());
      fo.y[0] = b.flogits;
      push(fo);
      Phase s{};
      s.op = OP_SAMPLE_FAST;
      s.cb = cb;
      push(s);
    }
  }

  // The Fast-AR-alone program (teacher-forced frames): the frame's hidden and first prefix code
  // (CTA 0), its projection into position 0, then the calls
  void fast_alone(const FastBufs& b, const FastWts& w) {
    new_program();
    Phase fi{};
    fi.op = OP_FAST_IN;
    push(fi);
    if (d.has_proj) {
      Phase p = gemv(d.Df, d.D, 1, w.P, nullptr, nullptr, EPI_STORE);
      p.col[0] = buf(b.hidden_src);
      p.y[0] = b.fx;
      push(p);
    } else {
      push(fi);  // a harmless repeat keeps the program length of every shape at 2 + the calls
    }
    fast_calls(b, w);
  }
};

}  // namespace

extern "C" {

int s2_weight_count(const s2_dims* s) {
  Dims d;
  std::string why;
  if (!s || !to_dims(s, d, why)) return -1;
  return layer_count(d);
}

long long s2_weight_info(const s2_dims* s, int i, char* name, int len) {
  Dims d;
  std::string why, nm;
  if (!s || !to_dims(s, d, why)) return -1;
  const long long n = tensor_numel(d, i, &nm);
  if (n >= 0 && name && len > 0) {
    std::snprintf(name, static_cast<size_t>(len), "%s", nm.c_str());
  }
  return n;
}

size_t s2_frame_workspace_bytes(const s2_dims* s, int max_streams, int kv_slots) {
  Dims d;
  std::string why;
  if (!s || !to_dims(s, d, why) || max_streams <= 0 || kv_slots < 0) return 0;
  s2_ctx tmp;
  tmp.d = d;
  tmp.max_streams = max_streams;
  tmp.kv_slots = d.L > 0 ? kv_slots : 0;
  int dev = 0;
  cudaGetDevice(&dev);
  int grid = 0;
  if (frame_kernel_grid(dev, &grid) != S2_OK) grid = 256;
  tmp.grid = grid;
  setup_batched(&tmp);
  Carver cv{nullptr};
  carve(&tmp, cv);
  return align_up(cv.off, 256);
}

}  // extern "C"

namespace {

FastBufs ctx_fast_bufs(s2_ctx* c, float* hidden_src) {
  FastBufs b{};
  b.hidden_src = hidden_src;
  b.fx = c->fx;
  b.fqkv = c->fqkv;
  b.fo = c->fo;
  b.fg = c->fg;
  b.fk = c->fk;
  b.fv = c->fv;
  b.flogits = c->flogits;
  b.fop = c->fop;
  b.fgp = c->fgp;
  b.fcode = c->fcode;
  return b;
}

int build_programs(s2_ctx* c) {
  const Dims& d = c->d;
  const size_t total = static_cast<size_t>(c->max_streams) * c->n_dec + c->n_fast;
  std::vector<Phase> all(total);
  Builder b{d, c->grid, all.data(), static_cast<int>(total)};
  b.add_tagged(c->x, 8ull * d.D);
  b.add_tagged(c->fx, 8ull * d.Wf * d.Df);
  b.add_tagged(c->gp, 8ull * std::max(d.F, 1));
  b.add_tagged(c->fgp, 16ull * d.Ff);
  b.add_tagged(c->qkv, 8ull * std::max((d.Hq + 2 * d.Hkv) * d.hd, 1));
  b.add_tagged(c->fqkv, 16ull * (d.Hqf + 2 * d.Hkvf) * d.hdf);
  const FastWts fw{c->fast.data(), c->P, c->FO, c->fnorm};
  for (int sid = 0; sid < c->max_streams && d.L > 0; ++sid) {
    const int before = b.n;
    b.new_program();
    float* hid = c->hidden + static_cast<size_t>(sid) * d.D;
    float* lg = c->logits + static_cast<size_t>(sid) * logits_stride(d);
    // 1. main draw on CTA 0 while the other CTAs project the hidden state into Fast-AR position 0
    if (d.has_proj) {
      Phase p = b.gemv(d.Df, d.D, 1, c->P, nullptr, nullptr, EPI_STORE);
      p.merge_main = 1;
      p.cta0 = 1;
      p.col[0] = Builder::buf(hid);
      p.y[0] = c->fx;
      b.push(p);
    } else {
      Phase p{};
      p.op = OP_SAMPLE_MAIN;
      b.push(p);
    }
    // 2. nine Fast-AR calls with their draws
    b.fast_calls(ctx_fast_bufs(c, hid), fw);
    // 3. Slow-AR step on [token, code_0..code_{NCB-1}]
    const size_t kvl = static_cast<size_t>(c->max_streams) * d.Hkv * c->kv_slots * d.hd * d.kvsz;
    const size_t kvs = static_cast<size_t>(sid) * d.Hkv * c->kv_slots * d.hd * d.kvsz;
    const int QKV = (d.Hq + 2 * d.Hkv) * d.hd;
    const float scale = static_cast<float>(1.0 / std::sqrt(static_cast<double>(d.hd)));
    for (int l = 0; l < d.L; ++l) {
      const LayerW& w = c->slow[l];
      Phase q = b.gemv(QKV, d.D, 1, w.wqkv, nullptr, w.an, EPI_STORE);
      q.col[0] = l == 0 ? GemvCol{SRC_EMBED, 0, c->st[sid].vals, c->x} : Builder::buf(c->x);
      q.y[0] = c->qkv;
      b.push(q, true);  // read only by the attention phase that follows, which polls its words
      Phase a{};
      a.op = OP_ATTN_SLOW;
      a.layer = l;
      a.qkv = c->qkv;
      a.out = c->o;
      if (b.use_planes()) a.outp = c->op;
      a.kc = c->kc + l * kvl + kvs;
      a.vc = c->vc + l * kvl + kvs;
      a.qn = w.qn;
      a.kn = w.kn;
      a.scale = scale;
      b.push(a);
      Phase o = b.gemv(d.D, d.Hq * d.hd, 1, w.wo, nullptr, nullptr, EPI_ADD);
      o.col[0] = b.use_planes() ? Builder::planes(c->op) : Builder::buf(c->o);
      o.y[0] = c->x;
      b.push(o);
      Phase u = b.gemv(d.F, d.D, 1, w.w1, w.w3, w.fn, EPI_SWIGLU);
      u.col[0] = Builder::buf(c->x);
      if (b.use_planes()) u.yp[0] = c->gp;
      else u.y[0] = c->g;
      b.push(u);
      Phase dn = b.gemv(d.D, d.F, 1, w.w2, nullptr, nullptr, EPI_ADD);
      dn.col[0] = b.use_planes() ? Builder::planes(c->gp) : Builder::buf(c->g);
      dn.y[0] = c->x;
      b.push(dn);
    }
    // final norm + tied logits on the admissible ids (sem_begin..sem_end contiguous, im_end last)
    Phase lo = b.gemv(d.A, d.D, 1, static_cast<const unsigned char*>(c->E) + static_cast<size_t>(d.sem_lo) * d.D * d.esz,
                      nullptr, c->norm, EPI_STORE);
    lo.last_row = static_cast<const unsigned char*>(c->E) + static_cast<size_t>(d.im_end) * d.D * d.esz;
    lo.col[0] = Builder::buf(c->x);
    lo.hid_out = hid;
    lo.y[0] = lg;
    lo.bump_pos = 1;
    b.push(lo);
    if (b.n - before != c->n_dec) return fail(c, S2_EINVAL, "internal: decode program length");
  }
  // Fast-AR-alone program (its own hidden and stream-state slots after the streams')
  {
    const int before = b.n;
    b.fast_alone(ctx_fast_bufs(c, c->hidden + static_cast<size_t>(c->max_streams) * d.D), fw);
    if (b.n - before != c->n_fast) return fail(c, S2_EINVAL, "internal: fast program length");
  }
  if (!b.err.empty()) return fail(c, S2_EINVAL, b.err);
  if (static_cast<size_t>(b.n) != total) return fail(c, S2_EINVAL, "internal: program length");
  std::string why;
  if (!planes_inside(all.data(), all.size(), c->ws, c->ws_bytes, why)) return fail(c, S2_EINVAL, "internal: " + why);
  if (cudaMemcpy(c->prog, all.data(), all.size() * sizeof(Phase), cudaMemcpyHostToDevice) != cudaSuccess)
    return fail(c, S2_ECUDA, "copying the phase programs failed");
  return S2_OK;
}

CallParams base_params(s2_ctx* c) {
  CallParams cp{};
  cp.d = c->d;
  cp.ctl = c->ctl;
  cp.part = c->part;
  cp.fcode = c->fcode;
  cp.flogits = c->flogits;
  cp.rope = c->rope;
  cp.rope_f = c->rope_f;
  cp.E = c->E;
  cp.CE = c->CE;
  cp.FE = c->FE;
  cp.kv_slots = c->kv_slots;
  cp.trace = c->trace;
  cp.trace_cap = c->trace_cap;
  cp.gbar_base = c->gbar_base;
  return cp;
}

}  // namespace

extern "C" {

int s2_frame_init(const s2_dims* s, const void* const* weights, int n_weights, void* workspace, size_t ws_bytes,
                  int max_streams, int kv_slots, s2_ctx** out) {
  if (!out) return fail(nullptr, S2_EINVAL, "out is NULL");
  *out = nullptr;
  Dims d;
  std::string why;
  if (!s || !to_dims(s, d, why)) return fail(nullptr, S2_EINVAL, "bad dims: " + why);
  if (max_streams <= 0 || max_streams > 1024) return fail(nullptr, S2_EINVAL, "max_streams must be in 1..1024");
  if (d.L > 0 && kv_slots <= 0) return fail(nullptr, S2_EINVAL, "kv_slots must be positive");
  if (!weights || n_weights != layer_count(d)) return fail(nullptr, S2_EINVAL, "weight table size does not match the dims");
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return fail(nullptr, S2_EINVAL, "workspace must be 256-byte aligned");
  for (int i = 0; i < n_weights; ++i) {
    const bool slow_part = i < 3 + 9 * d.L;
    const bool optional = (d.L == 0 && i < 3) || (i == 3 + 9 * d.L && !d.has_proj);
    if (!weights[i] && !optional) {
      std::string nm;
      tensor_numel(d, i, &nm);
      return fail(nullptr, S2_EINVAL, "missing weight " + nm);
    }
    if (weights[i] && (reinterpret_cast<uintptr_t>(weights[i]) & 15u))
      return fail(nullptr, S2_EINVAL, "weights must be 16-byte aligned");
    (void)slow_part;
  }
  s2_ctx* c = new s2_ctx();
  c->d = d;
  c->max_streams = max_streams;
  c->kv_slots = d.L > 0 ? kv_slots : 0;
  cudaGetDevice(&c->device);
  if (frame_kernel_grid(c->device, &c->grid) != S2_OK) {
    delete c;
    return fail(nullptr, S2_ECUDA, "the frame kernel cannot be resident on this device");
  }
  int i = 0;
  c->E = weights[i++];
  c->CE = weights[i++];
  c->norm = weights[i++];
  auto bind = [&](std::vector<LayerW>& v, int n) {
    v.resize(n);
    for (int l = 0; l < n; ++l) {
      LayerW& w = v[l];
      const void** f[9] = {&w.an, &w.wqkv, &w.qn, &w.kn, &w.wo, &w.fn, &w.w1, &w.w3, &w.w2};
      for (int k = 0; k < 9; ++k) *f[k] = weights[i++];
    }
  };
  bind(c->slow, d.L);
  c->P = weights[i++];
  c->FE = weights[i++];
  c->fnorm = weights[i++];
  c->FO = weights[i++];
  bind(c->fast, d.Lf);
  c->ws = static_cast<unsigned char*>(workspace);
  c->ws_bytes = ws_bytes;
  setup_batched(c);
  Carver cv{nullptr};
  carve(c, cv);
  if (align_up(cv.off, 256) > ws_bytes) {
    delete c;
    return fail(nullptr, S2_ENOMEM, "workspace too small: need " + std::to_string(align_up(cv.off, 256)) + " bytes");
  }
  if (d.fp8 && !c->batched) {
    std::string why;
    batch_supported(d, max_streams, &why);
    delete c;
    return fail(nullptr, S2_EINVAL, "fp8 weight streaming runs on the batched decode engine: " + why);
  }
  Carver real{c->ws};
  carve(c, real);
  // control block, stream states, tables
  Control ctl{};
  ctl.spin_limit = 2000000;
  if (cudaMemcpy(c->ctl, &ctl, sizeof(Control), cudaMemcpyHostToDevice) != cudaSuccess ||
      cudaMemset(c->st, 0, sizeof(StreamState) * (max_streams + 1)) != cudaSuccess ||
      // the tagged buffers start with tag 0, which no phase uses
      cudaMemset(c->x, 0, 8ull * d.D) != cudaSuccess || cudaMemset(c->fx, 0, 8ull * d.Wf * d.Df) != cudaSuccess ||
      cudaMemset(c->gp, 0, 8ull * std::max(d.F, 1)) != cudaSuccess || cudaMemset(c->fgp, 0, 16ull * d.Ff) != cudaSuccess ||
      cudaMemset(c->qkv, 0, 8ull * std::max((d.Hq + 2 * d.Hkv) * d.hd, 1)) != cudaSuccess ||
      cudaMemset(c->fqkv, 0, 16ull * (d.Hqf + 2 * d.Hkvf) * d.hdf) != cudaSuccess) {
    delete c;
    return fail(nullptr, S2_ECUDA, "initialising the workspace failed");
  }
  if (build_rope_tables(c->rope, c->kv_slots, d.hd, c->rope_f, d.Wf, d.hdf, d.rope_base, d.rope_bf16, nullptr) != S2_OK ||
      cudaDeviceSynchronize() != cudaSuccess) {
    delete c;
    return fail(nullptr, S2_ECUDA, "building the RoPE tables failed");
  }
  const int rc = build_programs(c);
  if (rc != S2_OK) {
    g_init_error = c->err;
    delete c;
    return rc;
  }
  c->host_pos.assign(max_streams, 0);
  c->host_prefilled.assign(max_streams, 0);
  if (d.fp8) {
    // quantise every projection once, and check the kernel's fp8 expansion on this device
    int bad = -1;
    bool ok = true;
    for (const QuantW& q : c->qw) ok = ok && quantize_e4m3(q.w, q.rows, q.cols, q.q, q.s, nullptr) == 0;
    ok = ok && e4m3_selfcheck(c->qbad, nullptr) == 0 &&
         cudaMemcpy(&bad, c->qbad, sizeof(int), cudaMemcpyDeviceToHost) == cudaSuccess;
    if (!ok || bad != 0) {
      delete c;
      return fail(nullptr, S2_ECUDA, !ok ? "quantising the projections to e4m3 failed"
                                         : "the fp8 expansion differs from the hardware conversion on this device");
    }
  }
  if (c->batched) {
    BatchModel& m = c->bm;
    m.d = d;
    m.qw = c->qw.data();
    m.n_qw = static_cast<int>(c->qw.size());
    m.E = c->E;
    m.CE = c->CE;
    m.FE = c->FE;
    m.P = d.has_proj ? c->P : nullptr;
    m.FO = c->FO;
    m.norm = c->norm;
    m.fnorm = c->fnorm;
    m.slow = c->slow.data();
    m.fast = c->fast.data();
    m.max_streams = max_streams;
    m.kv_slots = c->kv_slots;
    m.lstride = static_cast<int>(logits_stride(d));
    m.sms = c->sms;
    m.st = c->st;
    m.hidden = c->hidden;
    m.logits = c->logits;
    m.stage = c->stage;
    m.ctl = c->ctl;
    m.kc = c->kc;
    m.vc = c->vc;
    m.rope = c->rope;
    m.rope_f = c->rope_f;
    std::string why;
    c->batch = batch_create(m, &why);
    if (!c->batch) {
      g_init_error = "batched decode setup failed: " + why;
      delete c;
      return S2_ECUDA;
    }
  }
  *out = c;
  return S2_OK;
}

int s2_prefill(s2_ctx* c, int n, const int* ids, const int32_t* tokens, const int* lengths, CUstream_st* stream) {
  if (!c) return fail(nullptr, S2_EINVAL, "ctx is NULL");
  const Dims& d = c->d;
  if (d.L == 0) return fail(c, S2_ESTATE, "this context has no Slow-AR (Fast-AR-alone shape)");
  if (n <= 0 || !ids || !tokens || !lengths) return fail(c, S2_EINVAL, "bad prefill arguments");
  size_t off = 0;
  for (int k = 0; k < n; ++k) {
    const int sid = ids[k], T = lengths[k];
    if (sid < 0 || sid >= c->max_streams) return fail(c, S2_EINVAL, "stream id out of range");
    if (T <= 0) return fail(c, S2_EINVAL, "prompt length must be positive");
    if (T > c->kv_slots) return fail(c, S2_ECAPACITY, "prompt longer than the KV slots");
  }
  for (int k = 0; k < n; ++k) {
    const int sid = ids[k], T = lengths[k];
    PrefillArgs a{};
    a.d = d;
    a.E = c->E;
    a.CE = c->CE;
    a.norm = c->norm;
    a.layers = c->slow.data();
    a.tokens = tokens + off;
    a.T = T;
    a.chunk = c->prefill_chunk;
    const size_t kvl = static_cast<size_t>(c->max_streams) * d.Hkv * c->kv_slots * d.hd * d.kvsz;
    const size_t kvs = static_cast<size_t>(sid) * d.Hkv * c->kv_slots * d.hd * d.kvsz;
    a.kc0 = c->kc + kvs;
    a.vc0 = c->vc + kvs;
    a.kv_layer_stride = kvl;
    a.kv_slots = c->kv_slots;
    a.rope = c->rope;
    a.scratch = c->pscratch;
    a.hidden = c->hidden + static_cast<size_t>(sid) * d.D;
    a.logits = c->logits + static_cast<size_t>(sid) * logits_stride(d);
    a.st = c->st + sid;
    a.err = &c->ctl->error;
    a.tc = c->batch;
    a.tc_planes = c->pf_planes;
    a.tc_ld = c->pf_ld;
    a.tc_part = c->pf_part;
    const int rc = run_prefill(a, stream);
    if (rc != S2_OK) return fail(c, rc, std::string("prefill launch failed: ") + cudaGetErrorString(cudaGetLastError()));
    off += static_cast<size_t>(T) * (d.ncb + 1);
    c->host_pos[sid] = T;
    c->host_prefilled[sid] = 1;
  }
  return S2_OK;
}

int s2_stream_import(s2_ctx* c, int sid, int n_pos, const void* k, const void* v, const float* x_last,
                     CUstream_st* stream) {
  if (!c) return fail(nullptr, S2_EINVAL, "ctx is NULL");
  const Dims& d = c->d;
  if (d.L == 0) return fail(c, S2_ESTATE, "this context has no Slow-AR (Fast-AR-alone shape)");
  if (sid < 0 || sid >= c->max_streams) return fail(c, S2_EINVAL, "stream id out of range");
  if (n_pos <= 0) return fail(c, S2_EINVAL, "n_pos must be positive");
  if (n_pos > c->kv_slots) return fail(c, S2_ECAPACITY, "n_pos exceeds the KV slots");
  if (!k || !v || !x_last) return fail(c, S2_EINVAL, "null import pointer");
  if ((reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v)) % d.kvsz != 0 ||
      reinterpret_cast<uintptr_t>(x_last) % 4 != 0)
    return fail(c, S2_EINVAL, "import pointers are not aligned to their element size");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // cache layout: [layer][stream][KV head][slot][head_dim]; source: [layer][KV head][n_pos][head_dim]
  const size_t row = static_cast<size_t>(n_pos) * d.hd * d.kvsz;
  const size_t dpitch = static_cast<size_t>(c->kv_slots) * d.hd * d.kvsz;
  const size_t layer_dst = static_cast<size_t>(c->max_streams) * d.Hkv * dpitch;
  const size_t stream_dst = static_cast<size_t>(sid) * d.Hkv * dpitch;
  const size_t layer_src = static_cast<size_t>(d.Hkv) * row;
  for (int l = 0; l < d.L; ++l) {
    const size_t dst = l * layer_dst + stream_dst;
    if (cudaMemcpy2DAsync(c->kc + dst, dpitch, static_cast<const unsigned char*>(k) + l * layer_src, row, row,
                          d.Hkv, cudaMemcpyDeviceToDevice, s) != cudaSuccess ||
        cudaMemcpy2DAsync(c->vc + dst, dpitch, static_cast<const unsigned char*>(v) + l * layer_src, row, row,
                          d.Hkv, cudaMemcpyDeviceToDevice, s) != cudaSuccess)
      return fail(c, S2_ECUDA, std::string("KV import copy failed: ") + cudaGetErrorString(cudaGetLastError()));
  }
  const int rc = run_head(d, x_last, c->norm, c->E, c->hidden + static_cast<size_t>(sid) * d.D,
                          c->logits + static_cast<size_t>(sid) * logits_stride(d), c->st + sid, n_pos, stream);
  if (rc != S2_OK) return fail(c, rc, std::string("import head launch failed: ") + cudaGetErrorString(cudaGetLastError()));
  c->host_pos[sid] = n_pos;
  c->host_prefilled[sid] = 1;
  return S2_OK;
}

int s2_decode_frames(s2_ctx* c, int n, const int* ids, int n_frames, const s2_sampling* params, const float* expo,
                     const int32_t* forced, int32_t* codes, int32_t* n_out, const s2_debug_taps* taps,
                     CUstream_st* stream) {
  if (!c) return fail(nullptr, S2_EINVAL, "ctx is NULL");
  const Dims& d = c->d;
  if (d.L == 0) return fail(c, S2_ESTATE, "this context has no Slow-AR (Fast-AR-alone shape)");
  if (n <= 0 || !ids || !params || !expo || !codes || !n_out) return fail(c, S2_EINVAL, "bad decode arguments");
  if (n_frames <= 0 || n_frames > kMaxFramesPerCall) return fail(c, S2_EINVAL, "n_frames must be in 1..8192");
  for (int k = 0; k < n; ++k) {
    const int sid = ids[k];
    if (sid < 0 || sid >= c->max_streams) return fail(c, S2_EINVAL, "stream id out of range");
    if (!c->host_prefilled[sid]) return fail(c, S2_ESTATE, "stream not prefilled");
    if (c->host_pos[sid] + n_frames > c->kv_slots) return fail(c, S2_ECAPACITY, "decode would exceed the KV slots");
    const s2_sampling& p = params[k];
    if (p.top_k != kTopK) return fail(c, S2_EINVAL, "top_k must be 30");
    if (!(p.temperature > 0.f) || !(p.ras_temperature > 0.f)) return fail(c, S2_EINVAL, "temperatures must be > 0");
    if (!(p.top_p > 0.f && p.top_p <= 1.f) || !(p.ras_top_p > 0.f && p.ras_top_p <= 1.f))
      return fail(c, S2_EINVAL, "top_p must be in (0, 1]");
    if (p.ras_window < 1 || p.ras_window > kMaxWindow) return fail(c, S2_EINVAL, "ras_window must be in 1..16");
    for (int j = 0; j < k; ++j)
      if (ids[j] == sid) return fail(c, S2_EINVAL, "a stream appears twice");
  }
  if (c->batch && (n >= 2 || d.fp8)) {
    int max_ctx = 0;
    for (int k = 0; k < n; ++k) max_ctx = std::max(max_ctx, c->host_pos[ids[k]] + n_frames);
    std::string why;
    int rc = batch_decode(c->batch, n, ids, n_frames, params, expo, forced, taps, max_ctx, stream, &why);
    if (rc != S2_OK) return fail(c, rc, why);
    for (int k = 0; k < n; ++k) {
      const int sid = ids[k];
      rc = compact_codes(c->stage + static_cast<size_t>(sid) * kMaxFramesPerCall * d.ncb,
                         codes + static_cast<size_t>(k) * d.ncb * n_frames, c->st + sid, n_frames, d.ncb, n_out + k,
                         stream);
      if (rc != S2_OK) return fail(c, rc, "code compaction launch failed");
      c->host_pos[sid] += n_frames;
    }
    return S2_OK;
  }
  for (int k = 0; k < n; ++k) {
    const int sid = ids[k];
    CallParams cp = base_params(c);
    cp.n_frames = n_frames;
    cp.fast_only = 0;
    cp.n_phases = c->n_dec;
    cp.tag0 = take_tags(c->tag_next, static_cast<long long>(n_frames) * c->n_dec);
    cp.stream = sid;
    cp.prog = c->prog + static_cast<size_t>(sid) * c->n_dec;
    cp.st = c->st + sid;
    cp.hidden = c->hidden + static_cast<size_t>(sid) * d.D;
    cp.logits = c->logits + static_cast<size_t>(sid) * logits_stride(d);
    cp.stage = c->stage + static_cast<size_t>(sid) * kMaxFramesPerCall * d.ncb;
    const size_t fo = static_cast<size_t>(k) * n_frames;
    cp.expo = expo + fo * kDraws * kTopK;
    cp.forced = forced ? forced + fo * kDraws : nullptr;
    if (taps) {
      cp.dbg_main = taps->main_logits ? taps->main_logits + fo * d.A : nullptr;
      cp.dbg_fast = taps->fast_logits ? taps->fast_logits + fo * (d.ncb - 1) * d.cbs : nullptr;
      cp.dbg_hidden = taps->hidden ? taps->hidden + fo * d.D : nullptr;
      cp.dbg_draws = taps->draws ? taps->draws + fo * kDraws : nullptr;
    }
    const s2_sampling& p = params[k];
    cp.temperature = p.temperature;
    cp.top_p = p.top_p;
    cp.ras_temperature = p.ras_temperature;
    cp.ras_top_p = p.ras_top_p;
    cp.ras_window = p.ras_window;
    cp.min_tokens = p.min_tokens_before_end;
    // the kernel copies these with 16-byte (bulk or cp.async) copies
    if ((reinterpret_cast<uintptr_t>(cp.logits) | reinterpret_cast<uintptr_t>(cp.hidden) |
         reinterpret_cast<uintptr_t>(cp.flogits)) % 16 != 0)
      return fail(c, S2_EINVAL, "internal: a per-stream buffer is not 16-byte aligned");
    int rc = launch_frames(cp, c->grid, stream);
    if (rc != S2_OK) return fail(c, rc, std::string("frame kernel launch failed: ") + cudaGetErrorString(cudaGetLastError()));
    rc = compact_codes(cp.stage, codes + static_cast<size_t>(k) * d.ncb * n_frames, cp.st, n_frames, d.ncb, n_out + k,
                       stream);
    if (rc != S2_OK) return fail(c, rc, "code compaction launch failed");
    c->host_pos[sid] += n_frames;
  }
  return S2_OK;
}

int s2_stop_stream(s2_ctx* c, int sid, CUstream_st* side) {
  if (!c) return fail(nullptr, S2_EINVAL, "ctx is NULL");
  if (sid < 0 || sid >= c->max_streams) return fail(c, S2_EINVAL, "stream id out of range");
  static const int one = 1;
  if (cudaMemcpyAsync(&c->st[sid].stop_req, &one, sizeof(int), cudaMemcpyHostToDevice,
                      reinterpret_cast<cudaStream_t>(side)) != cudaSuccess)
    return fail(c, S2_ECUDA, std::string("stop request copy failed: ") + cudaGetErrorString(cudaGetLastError()));
  return S2_OK;
}

int s2_stream_progress(s2_ctx* c, int n, const int* ids, int32_t* out, CUstream_st* side) {
  if (!c) return fail(nullptr, S2_EINVAL, "ctx is NULL");
  if (n <= 0 || !ids || !out) return fail(c, S2_EINVAL, "bad progress arguments");
  for (int k = 0; k < n; ++k) {
    if (ids[k] < 0 || ids[k] >= c->max_streams) return fail(c, S2_EINVAL, "stream id out of range");
    if (cudaMemcpyAsync(out + k, &c->st[ids[k]].n_out, sizeof(int32_t), cudaMemcpyDeviceToHost,
                        reinterpret_cast<cudaStream_t>(side)) != cudaSuccess)
      return fail(c, S2_ECUDA, std::string("progress copy failed: ") + cudaGetErrorString(cudaGetLastError()));
  }
  return S2_OK;
}

int s2_fast_logits(s2_ctx* c, int n_frames, const float* hidden, const int32_t* prefix, float* logits,
                   CUstream_st* stream) {
  if (!c) return fail(nullptr, S2_EINVAL, "ctx is NULL");
  const Dims& d = c->d;
  if (n_frames <= 0 || n_frames > kMaxFastFrames || !hidden || !prefix || !logits)
    return fail(c, S2_EINVAL, "bad fast_logits arguments (n_frames must be in 1..1048576)");
  if (d.fp8) return fail(c, S2_ESTATE, "the Fast-AR-alone path streams bf16 weights (fp8 contexts decode frames only)");
  CallParams cp = base_params(c);
  cp.n_frames = n_frames;
  cp.fast_only = 1;
  cp.n_phases = c->n_fast;
  cp.tag0 = take_tags(c->tag_next, static_cast<long long>(n_frames) * c->n_fast);
  cp.prog = c->prog + static_cast<size_t>(c->max_streams) * c->n_dec;
  cp.st = c->st + c->max_streams;
  cp.hidden = c->hidden + static_cast<size_t>(c->max_streams) * d.D;
  cp.fin_hidden = hidden;
  cp.fin_prefix = prefix;
  cp.fout = logits;
  cp.temperature = 1.f;
  cp.top_p = 1.f;
  const int rc = launch_frames(cp, c->grid, stream);
  if (rc != S2_OK) return fail(c, rc, std::string("frame kernel launch failed: ") + cudaGetErrorString(cudaGetLastError()));
  return S2_OK;
}

int s2_sync_status(s2_ctx* c, CUstream_st* stream) {
  if (!c) return fail(nullptr, S2_EINVAL, "ctx is NULL");
  if (cudaStreamSynchronize(stream) != cudaSuccess)
    return fail(c, S2_ECUDA, std::string("stream synchronisation failed: ") + cudaGetErrorString(cudaGetLastError()));
  Control h;
  if (cudaMemcpy(&h, c->ctl, sizeof(Control), cudaMemcpyDeviceToHost) != cudaSuccess)
    return fail(c, S2_ECUDA, "reading the device status failed");
  if (h.error != 0) {
    const int z[3] = {0, 0, 0};
    cudaMemcpy(&c->ctl->error, z, sizeof(z), cudaMemcpyHostToDevice);
    if (h.error != S2_ETIMEOUT) return fail(c, h.error, "an input id was out of range");
    std::string msg = "a device-side wait gave up (site " + std::to_string(h.error_where);
    if (h.error_where != 10) {
      msg += ", CTA " + std::to_string(h.error_cta);
      if (h.error_phase >= 0) msg += ", phase " + std::to_string(h.error_phase) + " of the launch";
    }
    return fail(c, h.error, msg + ")");
  }
  return S2_OK;
}

int s2_set_spin_limit(s2_ctx* c, long long limit) {
  if (!c) return fail(nullptr, S2_EINVAL, "ctx is NULL");
  if (limit < 0) return fail(c, S2_EINVAL, "limit must be >= 0");
  const long long v = limit == 0 ? 2000000 : limit;
  if (cudaMemcpy(&c->ctl->spin_limit, &v, sizeof(v), cudaMemcpyHostToDevice) != cudaSuccess)
    return fail(c, S2_ECUDA, "setting the spin limit failed");
  return S2_OK;
}

int s2_set_barrier_base(s2_ctx* c, unsigned base) {
  if (!c) return fail(nullptr, S2_EINVAL, "ctx is NULL");
  c->gbar_base = base;
  return S2_OK;
}

int s2_set_trace(s2_ctx* c, unsigned long long* buf, int capacity) {
  if (!c) return fail(nullptr, S2_EINVAL, "ctx is NULL");
  if ((buf == nullptr) != (capacity == 0) || capacity < 0) return fail(c, S2_EINVAL, "bad trace buffer");
  c->trace = buf;
  c->trace_cap = capacity;
  return S2_OK;
}

int s2_phase_count(const s2_ctx* c, int fast_only) {
  if (!c) return -1;
  return fast_only ? c->n_fast : c->n_dec;
}

int s2_frame_free(s2_ctx* c) {
  if (c && c->batch) batch_destroy(c->batch);
  delete c;
  return S2_OK;
}

const char* s2_last_error(const s2_ctx* c) { return c ? c->err.c_str() : g_init_error.c_str(); }

}  // extern "C"

// ============================================ Fast-AR alone on static scratch (no allocation)
//
// s2_fast_logits_static serves callers that may not allocate device memory: a host application
// whose own memory pool has already reserved the device (a game engine, a DAW plug-in), or a
// latency-critical thread (an audio callback) that must not block in cudaMalloc/cudaFree.  Its
// scratch is a file-scope device array that is part of this library; every call on a device
// shares it.

namespace {

constexpr size_t kStaticScratchBytes = S2_STATIC_SCRATCH_BYTES;
constexpr int kStaticMaxPhases = 1024;
constexpr int kStaticMaxDevices = 64;
constexpr int kStaticMaxFrames = kMaxFastFrames;
constexpr int kStaticMaxWeights = 3 + 4 + 9 * 128;  // weight-table entries kept for the program key

// In host code this name is only a stand-in for the symbol: the device address of each device's
// copy comes from cudaGetSymbolAddress, made with that device current.
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

struct StaticDevice {
  unsigned char* scratch = nullptr;  // device address of g_static_scratch on this device
  int grid = 0;                      // frame kernel grid (one CTA per SM)
  // the program and RoPE table in the array were built for this shape and weight table
  bool have_prog = false;
  unsigned tag_next = 1;             // tag counter of the tagged handoffs on this device
  Dims d{};
  int n_weights = 0;
  const void* w[kStaticMaxWeights] = {};
};

std::mutex g_static_mu;                       // serialises the host side of the calls
StaticDevice g_static_dev[kStaticMaxDevices];
Phase g_static_prog[kStaticMaxPhases];        // host copy of the program being uploaded
LayerW g_static_layers[kStaticMaxPhases / 5]; // Fast-AR layers bound from the weight table

struct StaticLayout {
  Control* ctl;
  float2* rope_f;
  StreamState* st;
  FastBufs fb;
  Phase* prog;
};

// Scratch of the Fast-AR-alone program: the context's Fast-AR buffers, carved from the array.
size_t carve_static(const Dims& d, int n_phases, unsigned char* base, StaticLayout& s) {
  Carver cv{base};
  const int QKVf = (d.Hqf + 2 * d.Hkvf) * d.hdf;
  s.ctl = cv.take<Control>(1);
  s.rope_f = cv.take<float2>(static_cast<size_t>(d.Wf) * (d.hdf / 2));
  s.st = cv.take<StreamState>(1);
  FastBufs& b = s.fb;
  b.hidden_src = cv.take<float>(d.D);
  b.fx = cv.take<float>(2 * static_cast<size_t>(d.Wf) * d.Df);
  b.fqkv = cv.take<float>(4 * static_cast<size_t>(QKVf));
  b.fo = cv.take<float>(2 * static_cast<size_t>(d.Hqf) * d.hdf);
  b.fg = cv.take<float>(2 * static_cast<size_t>(d.Ff));
  b.fk = cv.take<float>(static_cast<size_t>(d.Lf) * d.Wf * d.Hkvf * d.hdf);
  b.fv = cv.take<float>(static_cast<size_t>(d.Lf) * d.Wf * d.Hkvf * d.hdf);
  b.flogits = cv.take<float>(d.cbs);
  b.fop = cv.take<uint16_t>(4 * static_cast<size_t>(d.Hqf) * d.hdf);
  b.fgp = cv.take<uint16_t>(8 * static_cast<size_t>(d.Ff));
  b.fcode = cv.take<int32_t>(16);
  s.prog = cv.take<Phase>(static_cast<size_t>(n_phases));
  return align_up(cv.off, 256);
}

// control block and stream state of a call: zero, with the default wait bound
__global__ void k_static_reset(Control* ctl, StreamState* st, long long spin_limit) {
  const int n = static_cast<int>(sizeof(Control) / sizeof(int));
  for (int i = threadIdx.x; i < n; i += blockDim.x) reinterpret_cast<int*>(ctl)[i] = 0;
  for (int i = threadIdx.x; i < static_cast<int>(sizeof(StreamState) / sizeof(int)); i += blockDim.x)
    reinterpret_cast<int*>(st)[i] = 0;
  __syncthreads();
  if (threadIdx.x == 0) ctl->spin_limit = spin_limit;
}

bool same_key(const StaticDevice& sd, const Dims& d, const void* const* w, int n) {
  if (!sd.have_prog || sd.n_weights != n || std::memcmp(&sd.d, &d, sizeof(Dims)) != 0) return false;
  for (int i = 0; i < n; ++i)
    if (sd.w[i] != w[i]) return false;
  return true;
}

int static_fail(int code, const std::string& msg) { return fail(nullptr, code, "s2_fast_logits_static: " + msg); }

}  // namespace

extern "C" int s2_fast_logits_static(const s2_dims* s, const void* const* weights, int n_weights, int n_frames,
                                     const float* hidden, const int32_t* prefix, float* logits, int32_t* status,
                                     CUstream_st* stream) {
  Dims d{};
  std::string why;
  if (!s || !to_dims(s, d, why)) return static_fail(S2_EINVAL, "bad dims: " + why);
  if (d.fp8) return static_fail(S2_EINVAL, "the static entry streams bf16 or fp32 weights (weight_fp8 must be 0)");
  if (!weights || n_weights != layer_count(d)) return static_fail(S2_EINVAL, "weight table size does not match the dims");
  if (n_frames <= 0 || n_frames > kStaticMaxFrames) return static_fail(S2_EINVAL, "n_frames must be in 1..1048576");
  if (!hidden || !prefix || !logits) return static_fail(S2_EINVAL, "hidden, prefix and logits are required");
  const int base = 3 + 9 * d.L;
  for (int i = base; i < n_weights; ++i) {
    if (i == base && !d.has_proj) continue;
    if (!weights[i]) return static_fail(S2_EINVAL, "a Fast-AR weight is NULL");
    if (reinterpret_cast<uintptr_t>(weights[i]) & 15u) return static_fail(S2_EINVAL, "weights must be 16-byte aligned");
  }
  const int n_phases = fast_alone_phases(d);
  if (n_phases > kStaticMaxPhases)
    return static_fail(S2_ENOMEM, "the Fast-AR program has " + std::to_string(n_phases) +
                                      " phases; the static path holds at most " + std::to_string(kStaticMaxPhases));
  StaticLayout probe{};
  const size_t need = carve_static(d, n_phases, nullptr, probe);
  if (need > kStaticScratchBytes)
    return static_fail(S2_ENOMEM, "this Fast-AR shape needs " + std::to_string(need) +
                                      " bytes of scratch; the static array holds " + std::to_string(kStaticScratchBytes));
  const int n_fast_w = n_weights - base;
  if (n_fast_w > kStaticMaxWeights) return static_fail(S2_ENOMEM, "too many Fast-AR weights for the static path");
  std::lock_guard<std::mutex> lock(g_static_mu);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return static_fail(S2_ECUDA, "no current CUDA device");
  if (dev < 0 || dev >= kStaticMaxDevices) return static_fail(S2_EINVAL, "device ordinal above 63");
  StaticDevice& sd = g_static_dev[dev];
  // the array's device address on this device, looked up on every call (this device is current):
  // after a device reset the module, and with it the array, is loaded again at a new address
  void* ptr = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&ptr, g_static_scratch);
  if (e != cudaSuccess) return static_fail(S2_ECUDA, std::string("cudaGetSymbolAddress failed: ") + cudaGetErrorString(e));
  if (sd.scratch != static_cast<unsigned char*>(ptr) || sd.grid == 0) {
    int grid = 0;
    if (frame_kernel_grid(dev, &grid) != S2_OK) return static_fail(S2_ECUDA, "the frame kernel cannot be resident on this device");
    sd = StaticDevice{};
    sd.grid = grid;
    sd.scratch = static_cast<unsigned char*>(ptr);
  }
  StaticLayout sl{};
  carve_static(d, n_phases, sd.scratch, sl);
  cudaStream_t cs = stream;
  if (!same_key(sd, d, weights + base, n_fast_w)) {
    // a new shape or weight table: build the program and the RoPE table into the array (the
    // program is copied from this library's host memory, which waits for the stream's earlier work)
    sd.have_prog = false;
    for (int l = 0; l < d.Lf; ++l) {
      const void* const* lw = weights + base + 4 + 9 * l;
      g_static_layers[l] = LayerW{lw[0], lw[1], lw[2], lw[3], lw[4], lw[5], lw[6], lw[7], lw[8]};
    }
    Builder b{d, sd.grid, g_static_prog, kStaticMaxPhases};
    b.add_tagged(sl.fb.fx, 8ull * d.Wf * d.Df);
    b.add_tagged(sl.fb.fgp, 16ull * d.Ff);
    b.add_tagged(sl.fb.fqkv, 16ull * (d.Hqf + 2 * d.Hkvf) * d.hdf);
    b.fast_alone(sl.fb, FastWts{g_static_layers, weights[base], weights[base + 3], weights[base + 2]});
    if (!b.err.empty()) return static_fail(S2_EINVAL, b.err);
    if (b.n != n_phases) return static_fail(S2_EINVAL, "internal: Fast-AR program length");
    if (!planes_inside(g_static_prog, static_cast<size_t>(b.n), sd.scratch, kStaticScratchBytes, why))
      return static_fail(S2_EINVAL, "internal: " + why);
    // the scratch starts from zero (the tagged buffers' tag 0 is used by no phase)
    if (cudaMemsetAsync(sd.scratch, 0, need, cs) != cudaSuccess)
      return static_fail(S2_ECUDA, "clearing the static scratch failed");
    if (cudaMemcpyAsync(sl.prog, g_static_prog, sizeof(Phase) * n_phases, cudaMemcpyHostToDevice, cs) != cudaSuccess)
      return static_fail(S2_ECUDA, "copying the program failed");
    if (build_rope_tables(nullptr, 0, d.hd, sl.rope_f, d.Wf, d.hdf, d.rope_base, d.rope_bf16, cs) != S2_OK)
      return static_fail(S2_ECUDA, "building the RoPE table failed");
    sd.have_prog = true;
    sd.d = d;
    sd.n_weights = n_fast_w;
    for (int i = 0; i < n_fast_w; ++i) sd.w[i] = weights[base + i];
  }
  // what must start from zero (the array keeps the previous call's contents)
  k_static_reset<<<1, 64, 0, cs>>>(sl.ctl, sl.st, 2000000);
  if (cudaGetLastError() != cudaSuccess) return static_fail(S2_ECUDA, "initialising the static scratch failed");
  CallParams cp{};
  cp.d = d;
  cp.ctl = sl.ctl;
  cp.fcode = sl.fb.fcode;
  cp.flogits = sl.fb.flogits;
  cp.rope_f = sl.rope_f;
  cp.FE = weights[base + 1];
  cp.n_frames = n_frames;
  cp.fast_only = 1;
  cp.n_phases = n_phases;
  cp.tag0 = take_tags(sd.tag_next, static_cast<long long>(n_frames) * n_phases);
  cp.prog = sl.prog;
  cp.st = sl.st;
  cp.hidden = sl.fb.hidden_src;
  cp.fin_hidden = hidden;
  cp.fin_prefix = prefix;
  cp.fout = logits;
  cp.temperature = 1.f;
  cp.top_p = 1.f;
  const int rc = launch_frames(cp, sd.grid, cs);
  if (rc != S2_OK) return static_fail(rc, std::string("frame kernel launch failed: ") + cudaGetErrorString(cudaGetLastError()));
  if (status && cudaMemcpyAsync(status, &sl.ctl->error, 2 * sizeof(int32_t), cudaMemcpyDeviceToDevice, cs) != cudaSuccess)
    return static_fail(S2_ECUDA, "copying the status failed");
  return S2_OK;
}
