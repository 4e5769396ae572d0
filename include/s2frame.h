/*
 * s2frame.h — C ABI of the GB300 (sm_103a) Dual-AR frame decoder for S2-Pro.
 *
 * One frame of the method, per stream (s2.cpp analysis ch.02 "Overall architecture and
 * Dual-AR data flow" §3.2-§3.5 and ch.06 "Fast-AR codebook decoding and the generation
 * main loop" §5.1):
 *   1. draw the main token from the Slow-AR logits + sem_mask (top-k 30 / top-p, draw =
 *      argmax(probs / E), E an exponential variate), redraw at (1.0, 0.9) when it repeats a
 *      token of the last 10 (RAS, ch.06 §6); stop on im_end;
 *   2. sem_code = clamp(token - sem_begin, 0, codebook_size - 1);
 *   3. nine Fast-AR calls (4-layer transformer over [fast_project_in·hidden ; fast_embeddings
 *      of the codes so far], positions from 0, causal, untied fast_output) each followed by a
 *      draw, giving codes 1..9 (ch.06 §1-§4);
 *   4. one Slow-AR step on [token, code_0..code_9] (36-layer GQA transformer with fp16 KV
 *      cache, q/k RMSNorm, RoPE base 1e6, SwiGLU, tied logits), producing the next logits and
 *      the normalised hidden state (ch.02 §3.2, §3.4).
 *
 * Conventions
 *  - Every call is asynchronous on the caller's CUDA stream; results are valid once that
 *    stream has been synchronised.  Calls on one context must be ordered (one stream, or
 *    synchronised between streams): they share the context's scratch memory.
 *  - "device" pointers are CUDA device memory (e.g. torch tensors); "host" pointers are
 *    ordinary host memory read before the call returns.
 *  - The library allocates no device memory: all of it (KV cache, per-stream state,
 *    scratch) lives in the caller's workspace.  It keeps a small host-side object and, for
 *    bf16 models, a private CUDA stream, the weights' tensor maps and one instantiated CUDA
 *    graph per stream count decoded together (released by s2_frame_free).
 *  - s2_stop_stream and s2_stream_progress are the exception to the ordering rule: they are
 *    meant to run on a second, non-blocking stream while a decode call is in flight.
 *  - Return values are S2_* status codes; no C++ exception crosses this boundary.  A
 *    message for the last failure is available from s2_last_error().
 *  - Problems detected on the device (a grid barrier or pipeline wait that gave up) are
 *    recorded in device memory and reported by s2_sync_status(); they never trap.
 */
#ifndef S2FRAME_H
#define S2FRAME_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st; /* a cudaStream_t; NULL means the legacy default stream */
typedef struct s2_ctx s2_ctx;

enum { S2_F32 = 0, S2_BF16 = 1, S2_F16 = 2 };

enum {
  S2_OK = 0,
  S2_EINVAL = 1,     /* bad argument or shape */
  S2_ENOMEM = 2,     /* workspace too small */
  S2_ECAPACITY = 3,  /* a stream would exceed its KV slots */
  S2_ECUDA = 4,      /* a CUDA runtime call failed */
  S2_ETIMEOUT = 5,   /* a device-side wait gave up (see s2_sync_status) */
  S2_ESTATE = 6      /* call not valid in the stream's state (e.g. not prefilled) */
};

/* Model shape (ch.02 §2 dims table; ch.04 "Model loading and GGUF" §2.2 hyper-parameters). */
typedef struct s2_dims {
  int dim, n_layer, n_head, n_kv_head, head_dim, ffn, vocab;
  int sem_begin, sem_end, im_end, n_codebooks, codebook_size;
  float sem_scale, norm_eps, rope_base;
  int qk_norm;          /* per-head RMSNorm of q and k before RoPE (must be 1 or 0) */
  int rope_table_bf16;  /* round the RoPE cos/sin table to bf16 */
  int fast_dim, fast_n_layer, fast_n_head, fast_n_kv_head, fast_head_dim, fast_ffn, fast_window,
      has_fast_project_in;
  int weight_dtype;     /* S2_F32 or S2_BF16: every weight tensor has this type */
  int kv_dtype;         /* Slow-AR KV cache element type: S2_F16 with bf16 weights, S2_F32 with fp32
                           weights (the supported pairs); head_dim == fast_head_dim, 64 or 128 */
  int weight_fp8;       /* 1: stream the projection matrices (wqkv, wo, w1, w3, w2 of both transformers,
                           fast_project_in, fast_output) as fp8 e4m3 with one fp32 scale per row
                           (scale = max|row| / 448, round to nearest even, saturating), quantised by
                           s2_frame_init into the workspace from the bf16 weights; embeddings, norms
                           and the tied logits stay bf16; activations stay fp32-exact (bf16 hi + lo
                           parts).  bf16 weights only, projection lengths multiples of 128, shapes
                           the batched decode supports (every decode runs there, n = 1 included;
                           s2_fast_logits is not available).  0: stream bf16. */
} s2_dims;

/* Sampler settings of one stream ([ch.06 §5.3, §6]; Mizuoto "Fish Speech" engine page:
 * top-k is fixed at 30). */
typedef struct s2_sampling {
  float temperature, top_p;          /* main and Fast-AR draws; temperature > 0, 0 < top_p <= 1 */
  float ras_temperature, ras_top_p;  /* repetition-aware redraw (1.0, 0.9 upstream) */
  int top_k;                         /* must be 30 */
  int ras_window;                    /* 1..10 recent tokens compared */
  int min_tokens_before_end;         /* im_end is masked while frames_done < this */
  int max_frames;                    /* informational; n_frames of each call bounds the loop */
} s2_sampling;

/* Optional per-frame debug outputs of s2_decode_frames (any member may be NULL). */
typedef struct s2_debug_taps {
  float* main_logits;   /* device [n][n_frames][codebook_size+1]: Slow-AR logits on the admissible
                           ids (sem_begin..sem_end, then im_end) used for the frame's main draw */
  float* fast_logits;   /* device [n][n_frames][n_codebooks-1][codebook_size] */
  float* hidden;        /* device [n][n_frames][dim]: normalised Slow-AR hidden given to Fast-AR */
  int32_t* draws;       /* device [n][n_frames][11]: the library's own outcome of each draw (main,
                           redraw, codebooks 1..9) before any forcing; -1 where not drawn */
} s2_debug_taps;

/* Weight table.  Order: embeddings [vocab][dim], codebook_embeddings [n_codebooks*codebook_size]
 * [dim], norm [dim]; per Slow-AR layer 9 tensors: attention_norm [dim], attention.wqkv
 * [(n_head+2*n_kv_head)*head_dim][dim] (rows q | k | v, head-major), attention.q_norm [head_dim],
 * attention.k_norm [head_dim], attention.wo [dim][n_head*head_dim], ffn_norm [dim],
 * feed_forward.w1 [ffn][dim], feed_forward.w3 [ffn][dim], feed_forward.w2 [dim][ffn]; then
 * fast_project_in [fast_dim][dim], fast_embeddings [codebook_size][fast_dim], fast_norm
 * [fast_dim], fast_output [codebook_size][fast_dim]; then 9 per Fast-AR layer as above with the
 * fast_* sizes.  Names follow the GGUF names of ch.04 §3.  All row-major. */
int s2_weight_count(const s2_dims* d);
/* Writes the i-th name (NUL-terminated, truncated to len) and returns its element count, or -1. */
long long s2_weight_info(const s2_dims* d, int i, char* name, int len);

/* Device bytes s2_frame_init needs for `max_streams` streams of `kv_slots` KV positions each. */
size_t s2_frame_workspace_bytes(const s2_dims* d, int max_streams, int kv_slots);

/* Validate the shape, bind the weight table (device pointers, caller-owned, must outlive the
 * context; entries of an absent part may be NULL: the Slow-AR tensors when n_layer == 0,
 * fast_project_in when has_fast_project_in == 0) and lay out the workspace (device, caller-owned,
 * >= s2_frame_workspace_bytes, 256-byte aligned).  Synchronous (builds tables on the device of
 * the current CUDA context).  Fast-AR entry checks of ch.06 §1 are enforced here: a fast decoder
 * must exist, and fast_window must cover n_codebooks positions. */
int s2_frame_init(const s2_dims* d, const void* const* weights, int n_weights, void* workspace,
                  size_t ws_bytes, int max_streams, int kv_slots, s2_ctx** out);

/* Prefill n streams (ids host [n]) with their prompts: tokens device int32, the streams'
 * [len][n_codebooks+1] matrices (column-major token layout of ch.02 §3.1: row 0 text/semantic
 * id, rows 1.. codes) concatenated in order; lengths host [n].  Resets each stream, writes KV
 * slots 0..len-1 and keeps the logits and normalised hidden of the last position. */
int s2_prefill(s2_ctx* ctx, int n, const int* stream_ids, const int32_t* tokens, const int* lengths,
               struct CUstream_st* stream);

/* Load one stream's decode state from caller memory instead of running s2_prefill (restoring a
 * saved stream).  The pages have no counterpart: their state after a prompt is the KV cache of
 * the Slow-AR (ch.02 §1: one fp16 slot per position and layer) plus the last position's output,
 * which is what this call takes.
 *   k, v    device [n_layer][n_kv_head][n_pos][head_dim] in the context's KV dtype (fp16 or
 *           fp32); position t of KV head g of layer l at ((l*n_kv_head + g)*n_pos + t)*head_dim
 *   x_last  device [dim] fp32: the Slow-AR residual of position n_pos-1 before the final norm
 * The call copies K/V into slots 0..n_pos-1 of the stream, computes the normalised hidden and
 * the admissible logits from x_last as s2_prefill does for its last position, and resets the
 * stream (window empty, no frames emitted).  The caller's buffers may be reused once the call's
 * work on `stream` has completed.  Errors: S2_EINVAL (bad id, n_pos <= 0, null or unaligned
 * pointer), S2_ECAPACITY (n_pos > kv_slots), S2_ESTATE (no Slow-AR), S2_ECUDA. */
int s2_stream_import(s2_ctx* ctx, int stream_id, int n_pos, const void* k, const void* v, const float* x_last,
                     struct CUstream_st* stream);

/* Decode up to n_frames frames for each of n prefilled streams (ids host [n]).
 *   params  host [n] sampler settings
 *   expo    device [n][n_frames][11][30] exponential variates E = -ln u (draw order: main,
 *           redraw, codebooks 1..9; index = rank within the top 30)
 *   forced  device [n][n_frames][11] or NULL: replaces the outcome of each draw (teacher forcing)
 *   codes   device [n][n_codebooks*n_frames]: stream i's block holds codes[cb*n_out_i + f]
 *           (ch.06 §8 layout, compacted to the frames actually produced)
 *   n_out   device [n]: frames produced (< n_frames when im_end was drawn)
 *   taps    host struct or NULL: debug outputs (see s2_debug_taps)
 * Streams resume where the previous call left them (KV, position, RAS window, logits).  Calls
 * with two or more streams on a bf16 context decode them together (one weight read per step);
 * the frame's kernel sequence is kept per stream count, so later calls with the same count
 * start without setup (continuous batching: re-form the batch between short calls). */
int s2_decode_frames(s2_ctx* ctx, int n, const int* stream_ids, int n_frames, const s2_sampling* params,
                     const float* expo, const int32_t* forced, int32_t* codes, int32_t* n_out,
                     const s2_debug_taps* taps, struct CUstream_st* stream);

/* Frame-level control while a decode call runs (ch.06 §7: a per-frame callback may cancel the
 * generation).  Both calls only enqueue a small copy on `side_stream`, which should be a
 * non-blocking stream other than the one running s2_decode_frames, so that the copy takes effect
 * (or is read) while that call is still running:
 *   s2_stop_stream      asks stream_id to stop at its next frame boundary; the frame is not
 *                       emitted, n_out of the running call counts the frames before it, and the
 *                       stream stays stopped until it is prefilled or imported again.
 *   s2_stream_progress  copies, for each of n stream ids (host array), the frames emitted so far
 *                       by the running (or last) call into out (host memory, int32 [n]; valid
 *                       once side_stream has completed the copy).
 * Errors: S2_EINVAL (bad id or pointer), S2_ECUDA. */
int s2_stop_stream(s2_ctx* ctx, int stream_id, struct CUstream_st* side_stream);
int s2_stream_progress(s2_ctx* ctx, int n, const int* stream_ids, int32_t* out, struct CUstream_st* side_stream);

/* Fast-AR alone, teacher-forced (ch.06 §1-§4): for each of n_frames frames, hidden device
 * [n_frames][dim] and prefix device [n_frames][n_codebooks-1] (code_0..code_{NCB-2}); writes
 * logits device [n_frames][n_codebooks-1][codebook_size], window w = 2..n_codebooks.
 * n_frames is in 1..1048576 (S2_EINVAL otherwise). */
int s2_fast_logits(s2_ctx* ctx, int n_frames, const float* hidden, const int32_t* prefix, float* logits,
                   struct CUstream_st* stream);

/* Synchronise `stream` and report device-side failures of earlier calls (S2_ETIMEOUT) or
 * S2_OK; clears the recorded failure.  After S2_ETIMEOUT, s2_last_error names the wait that gave
 * up first: its site, the CTA and the index of the phase in the launch's program.  Sites of the
 * persistent kernel: 1 grid barrier; 2 weight loader waiting for a free ring stage; 3 weight
 * loader draining its copies at exit; 4, 5 a projection waiting for its weight stage; 6 the bulk
 * copy of a projection input; 7 draining those copies; 8 a poll of tagged words.  Site 10: a wait
 * of the batched engine's kernels (no CTA or phase reported). */
int s2_sync_status(s2_ctx* ctx, struct CUstream_st* stream);

/* Testing hook: bound on device-side spin waits, in units of ~1 µs (0 restores the default of
 * about two seconds).  Lets a test make a wait give up without any fault. */
int s2_set_spin_limit(s2_ctx* ctx, long long limit);

/* Testing hook: value at which the device grid-barrier counter starts in later launches
 * (default 0).  The counter grows by the grid size at every phase and wraps around 2^32 in long
 * calls; a test starts it a few phases below 2^32 to exercise the wrap. */
int s2_set_barrier_base(s2_ctx* ctx, unsigned base);

/* Tracing hook: when buf (device, 2*capacity entries) is set, later decode / Fast-AR calls record,
 * for frame f and program phase p (index k = f*phase_count + p < capacity), the globaltimer (ns)
 * at which the first CTA's consumers leave phase p (buf[k]) and at which its weight producer has
 * issued all of phase p's tiles (buf[capacity + k]).  buf = NULL, capacity = 0 turns it off. */
int s2_set_trace(s2_ctx* ctx, unsigned long long* buf, int capacity);

/* Number of phases of one frame's program (fast_only: the Fast-AR-alone program), or -1. */
int s2_phase_count(const s2_ctx* ctx, int fast_only);

int s2_frame_free(s2_ctx* ctx);

/* Message of the last failure on this context (or, when ctx is NULL, of the last failed
 * s2_frame_init or s2_fast_logits_static); never NULL. */
const char* s2_last_error(const s2_ctx* ctx);

/* ---------------------------------------------------------------------------------------------
 * Fast-AR alone without a context or workspace: for callers that cannot allocate device memory.
 *
 * The pages describing the method have no counterpart of this call; it is a service of this
 * library only.  Some callers may not call cudaMalloc: a host application whose own memory pool
 * has already reserved the device memory (an allocation outside the pool fails or escapes its
 * accounting), or a latency-critical thread, such as an audio callback, that must not block in
 * cudaMalloc/cudaFree (they can synchronise the whole device).  Such a caller cannot provide the
 * workspace s2_frame_init needs.  This call computes what s2_fast_logits computes, with the same
 * kernel and the same phases, but its scratch (Fast-AR activations, within-frame K/V, RoPE table,
 * control block and phase program: about 0.8 MB at S2-Pro shapes) is a file-scope device array of
 * S2_STATIC_SCRATCH_BYTES that belongs to the library: every GPU on which the library's device code
 * is loaded holds it until the process exits.
 *
 *   d, weights, n_weights  the shape and the weight table of s2_frame_init (device pointers, 16-byte
 *                          aligned); only the Fast-AR part and fast_project_in are read, the other
 *                          entries may be NULL
 *   hidden   device [n_frames][dim] fp32; prefix device [n_frames][n_codebooks-1] int32
 *   logits   device [n_frames][n_codebooks-1][codebook_size] fp32 (output), windows 2..n_codebooks
 *   status   device int32 [2] or NULL (output): the device-detected result of this call, {S2_OK,
 *            S2_ETIMEOUT (a wait gave up) or S2_EINVAL (a prefix code outside 0..codebook_size-1),
 *            site}, written on `stream` after the kernel
 *
 * Allocates nothing: it calls no cudaMalloc, cudaFree or other allocating routine (the message of a
 * failed call is the one exception, on the host).  The caller owns every input and output.
 * Limits: the shape's scratch must fit S2_STATIC_SCRATCH_BYTES and its program 1024 phases, else
 * S2_ENOMEM and nothing is launched; n_frames in 1..1048576 (frames run one after another in the
 * same scratch, so their number does not grow it).
 * Set-up: the first call on a device (the current one) configures the kernel on that device; make
 * that first call before any stream capture.  The array is committed on a device when the
 * library's device code is loaded there: at this first call under lazy module loading (the CUDA
 * default), or when the library is loaded with CUDA_MODULE_LOADING=EAGER.  A caller whose memory
 * pool reserves the device should make its first call before the pool does.  Every call looks the
 * array's address up again (cudaGetSymbolAddress, no allocation once loaded), so a device reset
 * between calls only repeats the set-up.
 * Program: the first call with a given shape and weight table on a device (and the first call
 * after a call with another one) writes the phase program and the Fast-AR RoPE table into the
 * array; the program is copied from this library's host memory, so that call waits until the
 * stream's earlier work is done.  Later calls with the same shape and table launch only a small
 * reset kernel (control block and state to zero), the frame kernel and, with status, one
 * device-to-device copy, and never wait on the host.
 * Sharing: all calls on a device use the one array, which keeps the previous call's contents; each
 * call resets what must start from zero before its kernel.  Calls whose GPU work overlaps
 * (different streams, or host threads without ordering) race on the array and give undefined
 * results: issue them on one stream or synchronise between them.  The host side of concurrent
 * calls is serialised.
 * Errors (nothing launched): S2_EINVAL bad shape, pointer, alignment, count or device ordinal (> 63);
 * S2_ENOMEM above the limits; S2_ECUDA set-up, copy or launch failed.  Message: s2_last_error(NULL). */
#define S2_STATIC_SCRATCH_BYTES ((size_t)2 << 20)
int s2_fast_logits_static(const s2_dims* d, const void* const* weights, int n_weights, int n_frames,
                          const float* hidden, const int32_t* prefix, float* logits, int32_t* status,
                          struct CUstream_st* stream);

/* Codec quantizer decode, lookup-and-sum part (ch.02 §3.5: the 10 x T codes go through the
 * semantic VQ, quantizers.0, plus the sum of the residual VQs, quantizers.i, level by level):
 *   latent[f][e] = Σ_{cb = 0..n_codebooks-1} quantizer_cb[codes[cb * n_frames + f]][e]
 * summed in codebook order in fp32.  The upsampling that follows on the pages and the waveform
 * decoder are not part of this call.  Stateless; allocates nothing.
 *   quantizers  host array [n_codebooks] of device pointers, each bf16 [codebook_size][dim],
 *               16-byte aligned
 *   codes       device int32 [n_codebooks * n_frames] (the layout s2_decode_frames emits)
 *   latent      device fp32 [n_frames][dim]
 *   status      device int32 or NULL: S2_EINVAL is written there when a code is out of range
 *               (that codebook's term is left out of the frame)
 * Errors (nothing launched): S2_EINVAL bad counts (n_codebooks 1..16, dim a multiple of 8),
 * pointers or alignment; S2_ECUDA launch failed. */
int s2_codec_latent(int n_codebooks, int codebook_size, int dim, const void* const* quantizers, int n_frames,
                    const int32_t* codes, float* latent, int32_t* status, struct CUstream_st* stream);

/* e4m3 quantisation of bf16 rows, the one s2_frame_init applies to the projection matrices when
 * weight_fp8 = 1 (low-precision weight streaming; the precedent on the pages is s2.cpp's
 * K-quantised GGUF tensors, s2.cpp analysis ch.02 §5 and ch.04 §4; the e4m3 format and the row
 * scaling are this library's choice): per row r of w [rows][cols],
 *   scales[r] = max_k |w[r][k]| / 448          (fp32 division, rounded to nearest)
 *   codes[r][k] = e4m3(w[r][k] / scales[r])    (fp32 division; round to nearest, ties to even,
 *                                               saturating at ±448; never a NaN code)
 * and an all-zero row gets scale 0 and zero codes.  e4m3 = sign, 4 exponent bits (bias 7), 3
 * mantissa bits, exponent field 0 = subnormals m·2^-9.  The decode then uses
 * scales[r]·value(codes[r][k]) in place of w[r][k].
 *   w       device bf16 [rows][cols], 2-byte aligned
 *   codes   device uint8 [rows][cols]
 *   scales  device fp32 [rows], 4-byte aligned
 * Stateless; allocates nothing; asynchronous on `stream`.
 * Errors (nothing launched): S2_EINVAL bad pointer, alignment or size; S2_ECUDA launch failed. */
int s2_quantize_e4m3(const void* w, long long rows, int cols, uint8_t* codes, float* scales,
                     struct CUstream_st* stream);

/* The S2 draw on caller logits rows: the device routine both decode engines run (s2.cpp analysis
 * ch.06 §5 for the draw and the min_tokens masking of im_end; the Mizuoto "Fish Speech" engine
 * page for top-k fixed at 30 and winner = argmax(probs / -log u)).  For each row r:
 *   z = logits / temperature (fp32 division); entries that are not finite, and the im_end entry
 *   when block_end != 0, cannot be drawn;
 *   the top 30 by (z desc, id asc), -0 equal to +0; π = softmax over them (fp32, max-subtracted,
 *   summed in rank order); rank r is kept iff r == 0 or Σ_{s<r} π_s < top_p;
 *   out[r] = the id of the kept rank maximising π_r / E_r (ties -> the lower rank), or -1 when
 *   no entry of the row can be drawn.
 * Ids: sem_begin < 0 -> the entry index (Fast-AR codes); sem_begin >= 0 -> the admissible main
 * vocabulary of n = codebook_size + 1 entries: entry i < n - 1 is token sem_begin + i, entry
 * n - 1 is im_end.
 *   logits  device fp32 [rows][n], 4-byte aligned, n 1..4352
 *   expo    device fp32 [rows][30]: E of each rank (-log u, u uniform in (0, 1])
 *   out     device int32 [rows]
 * Stateless; allocates nothing; asynchronous on `stream`.
 * Errors (nothing launched): S2_EINVAL bad count, pointer or alignment, temperature not finite
 * or <= 0, top_p not finite; S2_ECUDA launch failed. */
int s2_draw(int rows, const float* logits, int n, int sem_begin, int im_end, int block_end, float temperature,
            float top_p, const float* expo, int32_t* out, struct CUstream_st* stream);

#ifdef __cplusplus
}
#endif
#endif /* S2FRAME_H */
