// Internal definitions of the frame engine shared by its translation units.
#pragma once

#include <cstddef>
#include <cstdint>
#include <string>

#include "../../include/s2frame.h"

namespace s2 {

// ---------------------------------------------------------------- constants

constexpr int kTopK = 30;              // fixed top-k (Mizuoto "Fish Speech" page)
constexpr int kDraws = 11;             // main, redraw, codebooks 1..9
constexpr int kMaxCodebooks = 15;      // vals[] holds NCB+1 <= 16 ids
constexpr int kMaxWindow = 16;         // RAS window capacity (ras_window <= 10 used)
constexpr int kMaxFramesPerCall = 8192;
constexpr int kMaxFastFrames = 1 << 20;        // Fast-AR-alone calls (teacher-forced frames)

// persistent frame kernel geometry
constexpr int kConsumerWarps = 8;
constexpr int kConsumers = 32 * kConsumerWarps;
constexpr int kThreads = kConsumers + 32;      // + one producer warp
constexpr int kStages = 4;                     // weight ring depth
constexpr int kStageBytes = 41216;             // one tile: 16 row segments of <= 1280 bf16 (+16 B pad each)
constexpr int kTileRows = 16;                  // rows per bf16 weight tile (the MMA m dimension)
constexpr int kTileRowPad = 16;                // bytes added to each tile row (bank-conflict-free ldmatrix)
constexpr int kXsBytes = 40960;                // shared activations: padded bf16 hi/lo rows of 1 column x <= 10232 (2 x <= 5112)
constexpr int kRedFloats = 2048;               // per-CTA partial sums (GEMV row × K-slice)
constexpr int kXRegFloats = 80;                // activation slice per lane held in registers
constexpr int kGemvChunksPerLane = 5;          // 16-byte chunks per lane: K-slices of 1/8 of <= 10240 bf16
constexpr int kAttnMaxChunk = 2048;            // workspace sizing of the split-K partials
constexpr int kAttnItemSlots = 64;             // target slots per Slow-AR attention split
constexpr int kAttnMaxSplits = 32;             // splits per KV head at most

enum Op : int {
  OP_GEMV = 1,       // y = W·normed(x) with epilogue; may carry a main draw on CTA 0
  OP_ATTN_SLOW,      // q/k norm + RoPE + KV store of the new slot + split-K attention + combine
  OP_ATTN_FAST,      // Fast-AR attention over the within-frame window
  OP_SAMPLE_FAST,    // one Fast-AR draw (CTA 0)
  OP_FAST_IN,        // Fast-AR-alone mode: load the frame's hidden and prefix (CTA 0)
  OP_SAMPLE_MAIN,    // main draw + redraw + RAS + clamp (CTA 0) when not merged into a GEMV
};

// GEMV column sources: an fp32 vector, the Slow-AR input embedding, a fast_embeddings row, or
// bf16 hi / lo rows (K each, hi + lo = the fp32 value to ~2^-17) written by the producing phase
enum Src : int { SRC_NONE = 0, SRC_BUF, SRC_EMBED, SRC_FEROW, SRC_PLANES };
enum Epi : int { EPI_STORE = 0, EPI_ADD, EPI_SWIGLU };

// --------------------------------------------------------------- the model

struct Dims {
  int D, L, Hq, Hkv, hd, F, V;
  int sem_lo, sem_hi, im_end, ncb, cbs;
  float sem_scale, eps;
  double rope_base;
  int qk_norm, rope_bf16;
  int Df, Lf, Hqf, Hkvf, hdf, Ff, Wf, has_proj;
  int wdt;       // S2_F32 / S2_BF16
  int kvdt;      // S2_F32 / S2_F16
  int esz;       // weight element bytes
  int kvsz;      // KV element bytes
  int A;         // admissible logits = cbs + 1
  int fp8;       // projection matrices streamed as e4m3 + per-row scales (quantised copies)
};

struct LayerW {
  const void *an, *wqkv, *qn, *kn, *wo, *fn, *w1, *w3, *w2;
};

// ------------------------------------------------------- device-side state

struct StreamState {
  int pos;           // KV slots filled
  int frames_done;   // frames emitted since prefill
  int done;          // im_end drawn
  int prefilled;
  int wlen;          // RAS window length
  int n_out;         // frames emitted by the current call
  int status;
  int stop_req;      // set by s2_stop_stream: stop at the next frame boundary
  int window[kMaxWindow];  // oldest first
  int vals[16];            // next Slow-AR input: [token, code_0..code_{NCB-1}]
};

struct Control {
  unsigned gbar;            // grid barrier counter (reset before each launch)
  int error;                // device-detected failure (S2_ETIMEOUT) of any launch
  int error_where;          // which wait gave up
  int error_cta;            // the CTA (frame kernel) whose wait gave up first
  long long spin_limit;     // wait bound in ~1 µs units
  int error_phase;          // that CTA's phase index within its launch (frame kernel; -1 unknown)
  int pad;
  unsigned tickets[64];     // split-K attention: arrivals per KV head
};

// ------------------------------------------------------------ the program

struct GemvCol {
  int src;            // Src
  int tag_back;       // 0: a plain buffer; n > 0: a tagged buffer written n phases earlier (see Phase)
  const void* p;      // SRC_BUF: float[K]; SRC_EMBED: int[NCB+1]; SRC_FEROW: int* code
  float* wb;          // nullable: CTA 0 writes the raw (pre-norm) column here
};

struct alignas(16) Phase {
  int op;
  int merge_main;     // OP_GEMV: CTA 0 performs the main draw instead of GEMV rows
  int cta0;           // first CTA doing GEMV rows
  int M, K, nmat, ncols, epi, rows_per_tile, Q;
  int Kt;                // bf16 weights: columns per tile (K = nkt * Kt), for every 16-row block
  int nkt;               //   and the count of K tiles
  // Tagged handoffs (bf16 models): the residual rows and the SwiGLU planes are written as 64-bit
  // words (value bits, then the writing phase's tag: the launch's base tag + the phase's index).
  // A reader of such a buffer polls for the tag of the phase that wrote it (GemvCol::tag_back)
  // instead of waiting at a grid barrier after that phase.
  int tag_out;           // y / yp / column write-backs of this phase are tagged words
  int no_sync;           // no grid barrier after this phase: the next one polls its tagged inputs
  const void* w[2];   // row-major [M][K]; w[1] is the gate partner for EPI_SWIGLU
  const void* last_row;  // nullable: source of row M-1 (admissible logits: im_end row)
  const void* normw;     // nullable RMSNorm weight [K]
  float* hid_out;        // nullable: CTA 0 writes normalised column 0 here
  GemvCol col[2];
  float* y[2];           // per-column output [M] (nullable when only planes are wanted)
  uint16_t* yp[2];       // nullable: per-column output as bf16 hi [M] then lo [M] rows
  // attention
  int layer, npos, pos0, cb;
  int bump_pos;          // CTA 0 advances the stream position after this phase
  int qkv_tag_back;      // attention: 0 = qkv holds floats; n > 0 = tagged words stored n phases earlier
  int rows_base, rows_rem;  // GEMV rows per CTA: the first rows_rem CTAs (after cta0) take rows_base + 1
  float scale;           // attention: 1/sqrt(head_dim)
  const float* qkv;      // [npos][QKV]
  float* out;            // [npos][Hq*hd]
  uint16_t* outp;        // nullable: the output as bf16 hi / lo rows, [npos][2][Hq*hd]
  void* kc;              // Slow: K cache of this layer/stream [Hkv][slots][hd]; Fast: [W][Hkv][hd] fp32
  void* vc;
  const void* qn;
  const void* kn;
};

struct alignas(16) CallParams {
  int n_frames;
  int fast_only;
  int n_phases;
  int stream;
  const Phase* prog;
  StreamState* st;
  float* hidden;          // [D] normalised Slow-AR hidden of the stream
  float* logits;          // [A] admissible Slow-AR logits of the stream
  int32_t* stage;         // [n_frames][NCB] emitted codes
  const float* expo;      // [n_frames][11][30]
  const int32_t* forced;  // [n_frames][11] or null
  float* dbg_main;        // [n_frames][A] or null
  float* dbg_fast;        // [n_frames][NCB-1][CBS] or null
  float* dbg_hidden;      // [n_frames][D] or null
  int32_t* dbg_draws;     // [n_frames][11] or null
  // Fast-AR alone
  const float* fin_hidden;    // [n_frames][D]
  const int32_t* fin_prefix;  // [n_frames][NCB-1]
  float* fout;                // [n_frames][NCB-1][CBS]
  // sampling
  float temperature, top_p, ras_temperature, ras_top_p;
  int ras_window, min_tokens;
  // scratch
  float* part;            // Slow-AR attention split-K partials: o [items][4][hd], then (m, l) [items][4]
  int32_t* fcode;         // [NCB] Fast-AR codes of the frame
  float* flogits;         // [CBS]
  const float2* rope;     // Slow-AR table [slots][hd/2]
  const float2* rope_f;   // Fast-AR table [Wf][hdf/2]
  Control* ctl;
  unsigned long long* trace;  // nullable: [frame][phase] consumer exit time, then producer issue-done time
  int trace_cap;              // entries per half
  Dims d;
  // weights for sampling / inputs
  const void* E;
  const void* CE;
  const void* FE;
  int kv_slots;
  unsigned gbar_base;     // grid-barrier counter value at launch (the launch sets it)
  unsigned tag0;          // tag of the launch's first phase (never 0; phase k: tag0 + k)
};

// host entry points between translation units
int launch_frames(const CallParams& cp, int grid, void* stream);
int frame_kernel_grid(int device, int* grid_out);
size_t frame_kernel_smem();
int build_rope_tables(float2* slow, int slots, int hd, float2* fast, int wf, int hdf, double base, int bf16,
                      void* stream);
int compact_codes(const int32_t* stage, int32_t* codes, const StreamState* st, int n_frames, int ncb,
                  int32_t* n_out, void* stream);

struct Batch;
struct PrefillArgs {
  Dims d;
  const void* E;
  const void* CE;
  const void* norm;
  const LayerW* layers;   // host array [L]
  const int32_t* tokens;  // device [T][NCB+1]
  int T;
  int chunk;
  void* kc0;              // K cache of layer 0 for this stream; layer stride = kv_layer_stride bytes
  void* vc0;
  size_t kv_layer_stride;
  int kv_slots;
  const float2* rope;
  float* scratch;         // chunk * per-position floats
  float* hidden;          // [D]
  float* logits;          // [A]
  StreamState* st;
  int* err;               // device word receiving S2_EINVAL on an out-of-range id
  // tensor-core projections (bf16 models): the projection kernel, planes and partials
  Batch* tc;
  uint16_t* tc_planes;    // [256][tc_ld]
  int tc_ld;
  float* tc_part;
};
int run_prefill(const PrefillArgs& a, void* stream);
// final norm + admissible logits of a residual x [D], then the stream reset to position pos
int run_head(const Dims& d, const float* x, const void* norm, const void* E, float* hidden, float* logits,
             StreamState* st, int pos, void* stream);
size_t prefill_scratch_floats(const Dims& d, int chunk);

// ------------------------------------------------------------- batched decode
// Several streams decoded together, every weight read once per step for the whole batch (bf16
// weights; see batch.cu).  The engine carves the buffers below from the workspace.

struct BatchSizes {
  size_t planes_rows;      // rows of each planes buffer (hi/lo of up to 2 * max_streams columns)
  int ldX, ldO, ldH;       // planes row lengths: projection inputs, attention outputs, SwiGLU outputs
  size_t part_floats;      // split-K partials
  size_t apart_floats;     // attention split partials
};

// e4m3 copy of one bf16 projection matrix (fp8 weight streaming)
struct QuantW {
  const void* w;      // the bf16 matrix it stands for
  uint8_t* q;         // codes [rows][cols]
  float* s;           // row scales [rows]
  long long rows;
  int cols;
};

struct BatchModel {
  Dims d;
  const QuantW* qw;        // [n_qw]: projections streamed as fp8 (none: bf16)
  int n_qw;
  const void *E, *CE, *FE, *P, *FO, *norm, *fnorm;
  const LayerW* slow;      // [L]
  const LayerW* fast;      // [Lf]
  int max_streams, kv_slots, lstride, sms;
  StreamState* st;
  float* hidden;
  float* logits;
  int32_t* stage;
  Control* ctl;
  unsigned char* kc;
  unsigned char* vc;
  const float2* rope;
  const float2* rope_f;
  uint16_t *pX, *pO, *pH;
  float *part, *bx, *bfx, *bfk, *bfv, *apart, *bflog;
  int32_t* bfcode;
  int* bctl;
  void* bstreams;          // device array of per-stream call settings
};

bool batch_supported(const Dims& d, int max_streams, std::string* why);
BatchSizes batch_sizes(const Dims& d, int max_streams, int sms);
size_t batch_stream_bytes(int max_streams);
struct Batch;
Batch* batch_create(const BatchModel& m, std::string* err);
void batch_destroy(Batch* b);
// Prompt projections on the same tensor-core kernel: columns = up to 128 prompt positions given
// as hi / lo planes [2*NC rows][ld]; writes split partials part[(z*splits + s)*NC + c][M]
// and returns the split count (-1 on error).
int batch_prefill_proj(Batch* b, const void* w0, const void* w1, int M, int K, const uint16_t* planes, int ld, int NC,
                       float* part, void* stream);
size_t batch_prefill_part_floats(const Dims& d, int sms);
// e4m3 codes and row scales of bf16 rows (rows x K): 0 or -1 (launch failed)
int quantize_e4m3(const void* w, long long rows, int K, uint8_t* q, float* scales, void* stream);
// the fp8 expansion of the projection kernel against the hardware conversion: *bad (device) =
// number of codes that differ
int e4m3_selfcheck(int* bad, void* stream);
// Prompt attention of a chunk (positions pos0..pos0+Tc-1, causal) on the tensor cores; K/V of this
// stream's layer [Hkv][slots][hd] fp16 already hold every slot up to pos0+Tc-1.  0 or -1.
int batch_prefill_attn(const float* QKV, int Tc, int pos0, const Dims& d, const void* Kc, const void* Vc, int slots,
                       float scale, float* O, void* stream);
constexpr int kPrefillChunkTC = 128;
// streams ids[0..n), n_frames frames; expo/forced/taps laid out as for s2_decode_frames
int batch_decode(Batch* b, int n, const int* ids, int n_frames, const s2_sampling* params, const float* expo,
                 const int32_t* forced, const s2_debug_taps* taps, int max_ctx, void* stream, std::string* err);

}  // namespace s2
