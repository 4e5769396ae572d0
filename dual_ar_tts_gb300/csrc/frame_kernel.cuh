// Persistent frame kernel: runs whole Dual-AR frames (main draw, nine Fast-AR calls with their
// draws, one Slow-AR step) for one stream in a single cooperative launch.
//
// Layout of a CTA (one per SM):
//   warp 8      producer: streams the CTA's weight tiles of every GEMV phase, in program order,
//               into a ring of shared-memory stages with 1-D bulk async copies (TMA engine).
//               Weights never depend on activations, so it runs ahead across grid barriers,
//               bounded only by ring capacity.
//   warps 0..7  consumers: execute the phase program; a grid barrier (bounded spin on a global
//               counter) separates dependent phases.
// Every wait is bounded; a wait that gives up records S2_ETIMEOUT in the control block and the
// whole grid leaves the kernel cleanly (no trap).
//
// The computations follow s2.cpp analysis ch.02 "Overall architecture and Dual-AR data flow"
// §3.2-§3.4 (input embedding, 36-layer block, tied logits, feedback), ch.06 "Fast-AR codebook
// decoding and the generation main loop" §1-§6 (Fast-AR window, causal mask offset 0, untied
// output, sem_mask, min_tokens_before_end, RAS, clamp) and the Mizuoto "Fish Speech" engine
// page (fp32 RMSNorm, adjacent-pair RoPE with a bf16 table, top-k 30, argmax(probs / -log u),
// draw order).
#pragma once
#include <cuda_runtime.h>

#include <type_traits>

#include "ptx.cuh"
#include "s2_internal.h"
#include "sampler.cuh"

namespace s2 {
// Internal linkage: every kernel instance unit compiles its own copy of the device code.
namespace {

// Compile-time configuration of one frame kernel: bf16 weights with an fp16 Slow-AR KV cache on
// the tensor cores, or fp32 weights with an fp32 cache on the CUDA cores; HD = head_dim of both
// transformers.  Each configuration is its own kernel, so that a kernel holds only the code it runs.
template <bool BF16, int HD>
struct Cfg {
  static constexpr bool bf16 = BF16;
  static constexpr int hd = HD;
  using KT = typename std::conditional<BF16, __half, float>::type;
};

constexpr int kMiscFloats = 64;

struct Smem {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t xsbar;   // bulk copies of a GEMV's activation planes into xs
  int abort_flag;   // consumers -> producer: stop streaming
  int fail;         // a consumer wait gave up: leave at the next phase boundary
  int sync_ok;
  int flag;
  int phase_k;      // the consumers' current phase index in the launch (failure reports)
  int pos_frame;    // the Slow-AR slot of the current frame (the stream position at the launch + f)
  int attn_ns, attn_chunk, attn_g, attn_s, attn_rep;  // the frame's Slow-AR attention plan (this CTA's item)
  const float* attn_pml;
  int fa_j, fa_h, fa_g, fa_rep;  // Fast-AR attention: this CTA's (position, head, KV head) item
  Phase ph[2];      // consumers: the current phase descriptor and the prefetched next one
  Phase pph[2];     // producer: the same, walked ahead of the consumers
  alignas(16) CallParams cp;         // the launch's parameters (shared, so that callees taking them by
                                     // reference do not need a per-thread local copy)
  float red[kRedFloats];             // GEMV partial sums
  float misc[kMiscFloats];           // GEMV sum-of-squares partials
  alignas(16) unsigned char xs[kXsBytes];  // GEMV activations | attention scratch | sampler scratch
  alignas(128) unsigned char ring[kStages][kStageBytes];
};
static_assert(sizeof(SampScratch) <= kXsBytes, "sampler scratch");

// misc[] regions
constexpr int kMiscSS = 0;                 // GEMV sum-of-squares partials [16]
// xs regions while a Slow-AR attention phase runs: K/V staging [2 rounds][RS slots][head_dim]
// (8 KB per buffer and operand), then fp32 scratch (float offsets)
constexpr int kXsStageBytes = 8192;                 // one round of K (or V) rows
constexpr int kXsQ = 4 * kXsStageBytes / 4;         // q heads of this CTA [4][128]
constexpr int kXsKV = kXsQ + 512;                   // new k, v [2][128] (fp32, as stored)
constexpr int kXsSc = kXsKV + 256;                  // scores / probabilities [4][64]
constexpr int kXsStat = kXsSc + 256;                // per head: alpha [4], m [4], l [4]; splits' (m, l) [4][32][2]
static_assert((kXsStat + 16 + 4 * kAttnMaxSplits * 2) * 4 <= kXsBytes, "attention scratch");

struct Pipe {
  int stage;
  uint32_t round;
  uint32_t xs_uses;  // completed uses of the xs barrier (its phase parity)
  uint32_t tag;      // tag of the phase being run (tagged handoffs, bf16 models)
  __device__ void advance() {
    if (++stage == kStages) {
      stage = 0;
      ++round;
    }
  }
};

// ------------------------------------------------------------------ helpers

__device__ __forceinline__ void rows_of(const Phase& ph, int cta, int G, int& r0, int& nr) {
  const int g2 = G - ph.cta0, i = cta - ph.cta0;
  if (i < 0 || g2 <= 0) {
    r0 = 0;
    nr = 0;
    return;
  }
  const int base = ph.rows_base, rem = ph.rows_rem;  // M / (G - cta0), M % (G - cta0), from the host
  r0 = i * base + (i < rem ? i : rem);
  nr = base + (i < rem ? 1 : 0);
}

// The first wait of a launch to give up records its site, CTA and the consumers' phase index.
__device__ __forceinline__ void record_timeout(const CallParams& cp, int phase, int where) {
  if (atomicCAS(&cp.ctl->error, 0, S2_ETIMEOUT) == 0) {
    cp.ctl->error_where = where;
    cp.ctl->error_cta = static_cast<int>(blockIdx.x);
    cp.ctl->error_phase = phase;
  }
}

// Bounded wait on an mbarrier phase; on give-up records the failure and returns false.
// try_wait suspends in hardware until the phase completes or a short time limit passes; the
// abort/failure flags (shared memory) are polled every 16 tries, the global error word and the
// clock every 256 tries, so the common case reacts to the completion without any global load.
__device__ __noinline__ bool wait_bar_slow(const CallParams& cp, Smem& S, uint64_t* bar, uint32_t parity, int where,
                                           bool producer) {
  long long t0 = -1;
  for (unsigned it = 1;; ++it) {
    if (mbar_test(bar, parity)) return true;
    if ((it & 15u) == 0) {
      if (producer ? (*reinterpret_cast<volatile int*>(&S.abort_flag) != 0)
                   : (*reinterpret_cast<volatile int*>(&S.fail) != 0))
        return false;
      if ((it & 255u) == 0) {
        if (ld_volatile_int(&cp.ctl->error) != 0) return false;
        const long long t = clock_us();
        if (t0 < 0) t0 = t;
        else if (t - t0 > cp.ctl->spin_limit) {
          record_timeout(cp, *reinterpret_cast<volatile int*>(&S.phase_k), where);
          return false;
        }
      }
    }
  }
}

__device__ __forceinline__ bool wait_bar(const CallParams& cp, Smem& S, uint64_t* bar, uint32_t parity, int where,
                                         bool producer) {
  if (mbar_test(bar, parity)) return true;
  return wait_bar_slow(cp, S, bar, parity, where, producer);
}

// Grid-wide barrier among the consumer threads of all CTAs.
__device__ bool grid_sync(const CallParams& cp, Smem& S, unsigned& target) {
  named_bar(1, kConsumers);
  target += gridDim.x;
  if (threadIdx.x == 0) {
    // a failed CTA leaves at once (its failure is already in the global error word); the global
    // error word itself is read only while waiting, off the path of the arrival
    int ok = *reinterpret_cast<volatile int*>(&S.fail) == 0;
    if (ok) {
      // release: this CTA's writes (ordered before by the named barrier) become visible with the
      // arrival; acquire on the spin makes every other CTA's writes visible after it
      red_release_add(&cp.ctl->gbar, 1u);
      const long long lim = cp.ctl->spin_limit;
      const long long t0 = clock_us();
      unsigned spins = 0;
      // the clock every 8 polls, the global error word every 64.  The counter may wrap around
      // 2^32 within a long call: the signed difference orders it correctly (it is never more
      // than one phase of arrivals away from the target)
      while (static_cast<int>(ld_acquire(&cp.ctl->gbar) - target) < 0) {
        if ((++spins & 7u) == 0) {
          if ((spins & 63u) == 0 && ld_volatile_int(&cp.ctl->error) != 0) {
            ok = 0;
            break;
          }
          if (clock_us() - t0 > lim) {
            record_timeout(cp, S.phase_k, 1);
            ok = 0;
            break;
          }
        }
      }
    }
    S.sync_ok = ok;
    if (!ok) S.fail = 1;
  }
  named_bar(1, kConsumers);
  return S.sync_ok != 0;
}

__device__ __forceinline__ void unpack16(const uint4& u, float* f, uint16_t) {
  f[0] = bf16lo(u.x); f[1] = bf16hi(u.x); f[2] = bf16lo(u.y); f[3] = bf16hi(u.y);
  f[4] = bf16lo(u.z); f[5] = bf16hi(u.z); f[6] = bf16lo(u.w); f[7] = bf16hi(u.w);
}
__device__ __forceinline__ void unpack16(const uint4& u, float* f, float) {
  f[0] = __uint_as_float(u.x); f[1] = __uint_as_float(u.y);
  f[2] = __uint_as_float(u.z); f[3] = __uint_as_float(u.w);
}

// v as bf16 hi (row 0, index i) and lo (row 1 at offset n): hi + lo = v to ~2^-17 relative
__device__ __forceinline__ void store_planes(uint16_t* planes, int n, int i, float v) {
  const float hi = bf16lo(cvt_bf16x2(v, 0.f));
  const uint32_t p = cvt_bf16x2(hi, v - hi);  // hi (exact) in the low half, lo in the high half
  planes[i] = static_cast<uint16_t>(p & 0xffffu);
  planes[n + i] = static_cast<uint16_t>(p >> 16);
}

// Split of the Slow-AR attention over n slots: ns splits of `chunk` slots per KV head, at most one
// item per CTA.
__device__ __forceinline__ void attn_split(int n, int G, int Hkv, int& ns, int& chunk) {
  ns = max(1, min(min(kAttnMaxSplits, max(1, G / Hkv)), (n + kAttnItemSlots - 1) / kAttnItemSlots));
  chunk = (n + ns - 1) / ns;
  ns = (n + chunk - 1) / chunk;
}
__device__ __forceinline__ const float* attn_part_ml(const CallParams& cp, int G) {
  return cp.part + static_cast<size_t>(cp.d.Hkv) * max(1, G / cp.d.Hkv) * 4 * cp.d.hd;
}

// Wait for bulk copies into this CTA's shared memory to land before it may leave the kernel.
// The bound is fixed (about two seconds, not the adjustable wait bound): copies complete within
// microseconds unless the memory system has failed.
constexpr long long kDrainLimitUs = 2000000;
__device__ __noinline__ void drain_copies(const CallParams& cp, uint64_t* bar, uint32_t parity, int where) {
  const long long t0 = clock_us();
  while (!mbar_test(bar, parity)) {
    if (clock_us() - t0 > kDrainLimitUs) {
      record_timeout(cp, -1, where);
      break;
    }
  }
}

// ---------------------------------------------------------------- tagged handoffs
// A tagged word holds a 32-bit value and, above it, the tag of the phase that stored it.  An
// aligned 8-byte store is single-copy atomic, so a reader that sees the tag it expects also sees
// that phase's value; it polls the words (L2, bypassing L1) instead of waiting at a grid barrier.
__device__ __forceinline__ unsigned long long tagw(uint32_t bits, uint32_t tag) {
  return (static_cast<unsigned long long>(tag) << 32) | bits;
}
// Polled words are read with relaxed loads at GPU scope (morally strong): a weak load in a polling
// loop has no visibility guarantee, and on this two-die part it was seen to keep returning a stale
// copy of a word for a second after the word had been stored.
__device__ __forceinline__ ulonglong2 ld_relaxed_u64x2(const unsigned long long* p) {
  ulonglong2 v;
  asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(v.x), "=l"(v.y) : "l"(p));
  return v;
}
__device__ __forceinline__ bool tags_are(const ulonglong2& a, uint32_t tag) {
  return static_cast<uint32_t>(a.x >> 32) == tag && static_cast<uint32_t>(a.y >> 32) == tag;
}
__device__ __forceinline__ float tval(unsigned long long w) { return __uint_as_float(static_cast<uint32_t>(w)); }

// Waits, bounded, until the pairs of tagged words at p[2i], p[2i + 1] (i in `miss`, a mask) carry
// `tag`; returns their values in v.  A give-up records S2_ETIMEOUT (site 8) and the CTA's failure.
template <int N>
__device__ __forceinline__ void wait_tagged(const CallParams& cp, Smem& S, const unsigned long long* const (&p)[N],
                                         uint32_t tag, uint32_t miss, ulonglong2 (&v)[N]) {
  const long long t0 = clock_us();
  for (unsigned it = 1; miss != 0u; ++it) {
#pragma unroll
    for (int i = 0; i < N; ++i)
      if (miss & (1u << i)) {
        v[i] = ld_relaxed_u64x2(p[i]);
        if (tags_are(v[i], tag)) miss &= ~(1u << i);
      }
    if (miss != 0u && (it & 15u) == 0u) {
      if (ld_volatile_int(&cp.ctl->error) != 0 || *reinterpret_cast<volatile int*>(&S.fail) != 0) break;
      if (clock_us() - t0 > cp.ctl->spin_limit) {
        record_timeout(cp, S.phase_k, 8);
        break;
      }
    }
  }
  if (miss != 0u) S.fail = 1;
}
// the same wait out of line (call sites whose registers are scarce: the attention phases)
template <int N>
__device__ __noinline__ void wait_tagged_nl(const CallParams& cp, Smem& S, const unsigned long long* const (&p)[N],
                                         uint32_t tag, uint32_t miss, ulonglong2 (&v)[N]) {
  const long long t0 = clock_us();
  for (unsigned it = 1; miss != 0u; ++it) {
#pragma unroll
    for (int i = 0; i < N; ++i)
      if (miss & (1u << i)) {
        v[i] = ld_relaxed_u64x2(p[i]);
        if (tags_are(v[i], tag)) miss &= ~(1u << i);
      }
    if (miss != 0u && (it & 15u) == 0u) {
      if (ld_volatile_int(&cp.ctl->error) != 0 || *reinterpret_cast<volatile int*>(&S.fail) != 0) break;
      if (clock_us() - t0 > cp.ctl->spin_limit) {
        record_timeout(cp, S.phase_k, 8);
        break;
      }
    }
  }
  if (miss != 0u) S.fail = 1;
}

// DPL consecutive values of an attention phase's projection input (element e of ph.qkv): plain
// floats, or tagged words of the projection phase (ph.qkv_tag_back > 0).  qkv_issue requests
// them; qkv_ready waits for any word not yet stored and unpacks the values.
template <int DPL>
struct QkvWords {
  ulonglong2 w[DPL / 2];
  const unsigned long long* p;
};
template <int DPL>
__device__ __forceinline__ void qkv_issue(const Phase& ph, size_t e, QkvWords<DPL>& t, float (&v)[DPL]) {
  if (ph.qkv_tag_back > 0) {
    t.p = reinterpret_cast<const unsigned long long*>(ph.qkv) + e;
#pragma unroll
    for (int i = 0; i < DPL / 2; ++i) t.w[i] = ld_relaxed_u64x2(t.p + 2 * i);
  } else {
#pragma unroll
    for (int j = 0; j < DPL; ++j) v[j] = ldcg(ph.qkv + e + j);
  }
}
template <int DPL>
__device__ __forceinline__ void qkv_ready(const CallParams& cp, Smem& S, const Phase& ph, uint32_t tag,
                                          QkvWords<DPL>& t, float (&v)[DPL]) {
  if (ph.qkv_tag_back <= 0) return;
  const uint32_t want = tag - static_cast<uint32_t>(ph.qkv_tag_back);
  uint32_t miss = 0u;
#pragma unroll
  for (int i = 0; i < DPL / 2; ++i)
    if (!tags_are(t.w[i], want)) miss |= 1u << i;
  if (miss != 0u) {
    const unsigned long long* ptr[DPL / 2];
#pragma unroll
    for (int i = 0; i < DPL / 2; ++i) ptr[i] = t.p + 2 * i;
    wait_tagged_nl<DPL / 2>(cp, S, ptr, want, miss, t.w);
  }
#pragma unroll
  for (int i = 0; i < DPL / 2; ++i) {
    v[2 * i] = tval(t.w[i].x);
    v[2 * i + 1] = tval(t.w[i].y);
  }
}

// an output row of the phase's column c (read back for a residual add): tagged word or float
__device__ __forceinline__ float ld_out(const Phase& ph, int c, int row) {
  return ph.tag_out ? tval(__ldcg(reinterpret_cast<const unsigned long long*>(ph.y[c]) + row)) : ldcg(ph.y[c] + row);
}

// =========================================================================
// producer
// =========================================================================

// Producer warp: walks the program ahead of the consumers and fills the ring with each GEMV
// phase's weights (the RMSNorm vector first, then the row tiles).  Lane 0 waits for a free stage
// and posts the byte count; the tile's row segments are then issued by separate lanes.
__device__ bool producer_acquire(const CallParams& cp, Smem& S, Pipe& pp, uint32_t bytes) {
  const int lane = threadIdx.x & 31;
  int ok = 1;
  if (lane == 0) {
    ok = wait_bar(cp, S, &S.empty[pp.stage], (pp.round & 1u) ^ 1u, 2, true) ? 1 : 0;
    if (ok) mbar_arrive_expect_tx(&S.full[pp.stage], bytes);
  }
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

template <class C>
__device__ void producer(const CallParams& cp, Smem& S) {
  const int lane = threadIdx.x & 31;
  constexpr int NQ = static_cast<int>(sizeof(Phase) / 16);
  static_assert(NQ <= 32, "one 16-byte piece of a phase descriptor per producer lane");
  const uint64_t pol = policy_evict_first();
  Pipe pp{0, 0, 0, 0u};
  unsigned long long issued = 0;  // stages filled so far (all lanes keep the same count)
  int stop = (ld_volatile_int(&cp.st->done) != 0 && !cp.fast_only) ? 1 : 0;
  if (lane < NQ) reinterpret_cast<uint4*>(&S.pph[0])[lane] = __ldg(reinterpret_cast<const uint4*>(cp.prog) + lane);
  __syncwarp();
  int k = 0;
  for (int f = 0; f < cp.n_frames && !stop; ++f) {
    for (int p = 0; p < cp.n_phases && !stop; ++p, ++k) {
      const Phase& ph = S.pph[k & 1];
      const int np = (p + 1 == cp.n_phases) ? 0 : p + 1;
      const bool has_next = (p + 1 < cp.n_phases) || (f + 1 < cp.n_frames);
      uint4 nx = make_uint4(0u, 0u, 0u, 0u);
      if (lane < NQ && has_next) nx = __ldg(reinterpret_cast<const uint4*>(cp.prog + np) + lane);
      if (ph.op == OP_GEMV && !(ph.merge_main && blockIdx.x == 0)) {
        int r0, nr;
        rows_of(ph, blockIdx.x, gridDim.x, r0, nr);
        const uint32_t rowb = static_cast<uint32_t>(ph.K) * cp.d.esz;
        if (ph.normw != nullptr) {
          // the RMSNorm weight vector travels through the ring ahead of the phase's row tiles
          if (!producer_acquire(cp, S, pp, rowb)) {
            stop = 1;
          } else {
            if (lane == 0) bulk_g2s(S.ring[pp.stage], ph.normw, rowb, &S.full[pp.stage], pol);
            pp.advance();
            ++issued;
          }
        }
        if constexpr (C::bf16) {
          // bf16: tiles of <= 8 rows x Kt columns, row segments padded by 16 bytes, one lane per row
          for (int b = 0; b < nr && !stop; b += kTileRows) {
            const int rows = min(kTileRows, nr - b);
            // the phase's 16-row K tiling (no per-block division on the issue path); a short last
            // block whose rows fit one stage whole takes all of K in one tile
            int Kt = ph.Kt, nkt = ph.nkt;
            if (rows < kTileRows && rows * (2 * ph.K + kTileRowPad) <= kStageBytes) {
              Kt = ph.K;
              nkt = 1;
            }
            const uint32_t segb = static_cast<uint32_t>(Kt) * 2u, pitch = segb + kTileRowPad;
            const int row = r0 + b + lane;
            for (int m = 0; m < ph.nmat && !stop; ++m) {
              const unsigned char* rsrc =
                  (ph.last_row != nullptr && row == ph.M - 1)
                      ? static_cast<const unsigned char*>(ph.last_row)
                      : static_cast<const unsigned char*>(ph.w[m]) + static_cast<size_t>(row) * rowb;
              for (int kt = 0; kt < nkt; ++kt) {
                if (!producer_acquire(cp, S, pp, segb * rows)) {
                  stop = 1;
                  break;
                }
                if (lane < rows)
                  bulk_g2s(S.ring[pp.stage] + lane * pitch, rsrc + static_cast<size_t>(kt) * segb, segb,
                           &S.full[pp.stage], pol);
                pp.advance();
                ++issued;
              }
            }
          }
        } else {
          // fp32: tiles of whole rows, one copy
          const int R = ph.rows_per_tile;
          for (int t = 0; t < nr && !stop; t += R) {
            const int rr = min(R, nr - t);
            if (!producer_acquire(cp, S, pp, rowb * rr * ph.nmat)) {
              stop = 1;
              break;
            }
            if (lane < ph.nmat) {
              const unsigned char* src =
                  static_cast<const unsigned char*>(ph.w[lane]) + static_cast<size_t>(r0 + t) * rowb;
              unsigned char* dm = S.ring[pp.stage] + static_cast<size_t>(lane) * rr * rowb;
              if (ph.last_row != nullptr && r0 + t + rr == ph.M) {
                if (rr > 1) bulk_g2s(dm, src, rowb * (rr - 1), &S.full[pp.stage], pol);
                bulk_g2s(dm + static_cast<size_t>(rr - 1) * rowb, ph.last_row, rowb, &S.full[pp.stage], pol);
              } else {
                bulk_g2s(dm, src, rowb * rr, &S.full[pp.stage], pol);
              }
            }
            pp.advance();
            ++issued;
          }
        }
        if (lane == 0 && cp.trace != nullptr && blockIdx.x == 0) {
          const int kk = f * cp.n_phases + p;
          if (kk < cp.trace_cap) cp.trace[cp.trace_cap + kk] = globaltimer_ns();
        }
      }
      stop = __shfl_sync(0xffffffffu, stop, 0);
      if (lane < NQ && has_next) reinterpret_cast<uint4*>(&S.pph[(k + 1) & 1])[lane] = nx;
      __syncwarp();
    }
  }
  if (lane != 0) return;
  // Leave no copy in flight: the last fill of each stage must have landed before the CTA exits.
  for (unsigned long long back = 1; back <= kStages && back <= issued; ++back) {
    const unsigned long long t = issued - back;
    drain_copies(cp, &S.full[static_cast<int>(t % kStages)], static_cast<uint32_t>((t / kStages) & 1u), 3);
  }
}

// =========================================================================
// GEMV phase:  y[c][r] = W[r,:] · xn[c]   (xn = RMSNorm(x)·normw, or x)
// =========================================================================

template <typename WT, int NC>
__device__ __noinline__ Pipe gemv_t(const CallParams& cp, const Phase& ph, Smem& S, Pipe pipe) {
  constexpr int EPC = 16 / static_cast<int>(sizeof(WT));
  constexpr int NCH = kGemvChunksPerLane;  // every warp holds a 1/8 K-slice: <= 5 chunks per lane
  const Dims& d = cp.d;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int K = ph.K, Q = ph.Q;
  const int nchunk = K / EPC;
  const int slice = (nchunk + Q - 1) / Q;
  const int q = warp % Q, group = warp / Q;
  const int c_beg = q * slice, c_end = min(nchunk, c_beg + slice);
  const bool writer = (blockIdx.x == 0) && (group == 0);
  const bool has_norm = ph.normw != nullptr;
  int r0, nr;
  rows_of(ph, blockIdx.x, gridDim.x, r0, nr);
  // the residual rows of an accumulate phase are final since an earlier phase: request them now
  float yres = 0.f;
  if (ph.epi == EPI_ADD && tid < nr * NC) yres = ldcg(ph.y[tid % NC] + r0 + tid / NC);

  // ---- resolve each column's source: fp32 global vector, weight row (bf16/fp32), or the
  // Slow-AR input embedding, which is summed here into shared memory first
  const float* xf[NC];
  const unsigned char* xw[NC];
  bool staged = false;
#pragma unroll
  for (int c = 0; c < NC; ++c) {
    const GemvCol col = ph.col[c];
    xf[c] = nullptr;
    xw[c] = nullptr;
    if (col.src == SRC_BUF) {
      xf[c] = static_cast<const float*>(col.p);
    } else if (col.src == SRC_FEROW) {
      const int code = ldcgi(static_cast<const int*>(col.p));
      xw[c] = static_cast<const unsigned char*>(cp.FE) + static_cast<size_t>(code) * K * sizeof(WT);
    } else {
      // x = sem_scale·E[r0] + m·Σ_cb CE[cb·CBS + code_cb], m = [r0 semantic]   (ch.02 §3.2)
      const int* vals = static_cast<const int*>(col.p);
      const int tok = ldcgi(vals);
      const float m = (tok >= d.sem_lo && tok <= d.sem_hi) ? 1.f : 0.f;
      float* xs = S.red + c * K;
      for (int e = tid; e < K; e += kConsumers) {
        float acc = 0.f;
        for (int cb = 0; cb < d.ncb; ++cb) {
          const size_t row = static_cast<size_t>(cb) * d.cbs + ldcgi(vals + 1 + cb);
          acc = __fadd_rn(acc, wload(cp.CE, row * K + e, sizeof(WT)));
        }
        xs[e] = __fadd_rn(__fmul_rn(d.sem_scale, wload(cp.E, static_cast<size_t>(tok) * K + e, sizeof(WT))),
                          __fmul_rn(m, acc));
      }
      xf[c] = xs;
      staged = true;
    }
  }
  if (staged) named_bar(1, kConsumers);

  // ---- activation slices into registers (all loads issued before any store)
  float xr[NC][NCH][EPC];
#pragma unroll
  for (int c = 0; c < NC; ++c) {
#pragma unroll
    for (int i = 0; i < NCH; ++i)
#pragma unroll
      for (int j = 0; j < EPC; ++j) xr[c][i][j] = 0.f;
    if (xw[c] != nullptr) {
#pragma unroll
      for (int i = 0; i < NCH; ++i) {
        const int ch = c_beg + lane + 32 * i;
        if (ch < c_end) unpack16(ldnc_u4(xw[c] + static_cast<size_t>(ch) * 16), xr[c][i], WT());
      }
    } else if (staged) {
#pragma unroll
      for (int i = 0; i < NCH; ++i) {
        const int ch = c_beg + lane + 32 * i;
        if (ch < c_end)
#pragma unroll
          for (int j = 0; j < EPC; j += 4) {
            const float4 v = *reinterpret_cast<const float4*>(xf[c] + ch * EPC + j);
            xr[c][i][j] = v.x; xr[c][i][j + 1] = v.y; xr[c][i][j + 2] = v.z; xr[c][i][j + 3] = v.w;
          }
      }
    } else {
#pragma unroll
      for (int i = 0; i < NCH; ++i) {
        const int ch = c_beg + lane + 32 * i;
        if (ch < c_end)
#pragma unroll
          for (int j = 0; j < EPC; j += 4) {
            const float4 v = ldcg4(xf[c] + ch * EPC + j);
            xr[c][i][j] = v.x; xr[c][i][j + 1] = v.y; xr[c][i][j + 2] = v.z; xr[c][i][j + 3] = v.w;
          }
      }
    }
  }
  // raw (pre-norm) column written back for the residual stream (one CTA, one copy of each slice)
  if (writer) {
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      float* wb = ph.col[c].wb;
      if (wb == nullptr) continue;
#pragma unroll
      for (int i = 0; i < NCH; ++i) {
        const int ch = c_beg + lane + 32 * i;
        if (ch < c_end)
#pragma unroll
          for (int j = 0; j < EPC; j += 4)
            *reinterpret_cast<float4*>(wb + ch * EPC + j) = make_float4(xr[c][i][j], xr[c][i][j + 1], xr[c][i][j + 2], xr[c][i][j + 3]);
      }
    }
  }

  // ---- RMSNorm (fp32): each slice is held once by the warps of group 0
  if (has_norm) {
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      float ss = 0.f;
#pragma unroll
      for (int i = 0; i < NCH; ++i)
#pragma unroll
        for (int j = 0; j < EPC; ++j) ss += xr[c][i][j] * xr[c][i][j];
      ss = warp_sum(ss);
      if (group == 0 && lane == 0) S.misc[kMiscSS + q * NC + c] = ss;
    }
  }
  named_bar(1, kConsumers);
  if (has_norm) {
    // the norm weights are the phase's first ring stage
    const bool ok = wait_bar(cp, S, &S.full[pipe.stage], pipe.round & 1u, 5, false);
    if (!ok) S.fail = 1;
    const unsigned char* nws = S.ring[pipe.stage];
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      float tot = 0.f;
      for (int qq = 0; qq < Q; ++qq) tot += S.misc[kMiscSS + qq * NC + c];
      const float r = 1.0f / sqrtf(tot / static_cast<float>(K) + d.eps);
#pragma unroll
      for (int i = 0; i < NCH; ++i) {
        const int ch = c_beg + lane + 32 * i;
        if (ch < c_end) {
          float wv[EPC];
          unpack16(*reinterpret_cast<const uint4*>(nws + static_cast<size_t>(ch) * 16), wv, WT());
#pragma unroll
          for (int j = 0; j < EPC; ++j) xr[c][i][j] = (xr[c][i][j] * r) * wv[j];
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.empty[pipe.stage]);
    pipe.advance();
    if (writer && ph.hid_out != nullptr) {
#pragma unroll
      for (int i = 0; i < NCH; ++i) {
        const int ch = c_beg + lane + 32 * i;
        if (ch < c_end)
#pragma unroll
          for (int j = 0; j < EPC; j += 4)
            *reinterpret_cast<float4*>(ph.hid_out + ch * EPC + j) =
                make_float4(xr[0][i][j], xr[0][i][j + 1], xr[0][i][j + 2], xr[0][i][j + 3]);
      }
    }
  }

  // ---- stream the CTA's row tiles: all eight warps work on every tile, each on its K-slice of
  // every row, four rows at a time (independent accumulation chains)
  const int R = ph.rows_per_tile;
  const int nmat = ph.nmat;
  const size_t rowb = static_cast<size_t>(K) * sizeof(WT);
  const int ntiles = (nr + R - 1) / R;
  for (int t = 0; t < ntiles; ++t) {
    const int rr = min(R, nr - t * R);
    const bool ok = wait_bar(cp, S, &S.full[pipe.stage], pipe.round & 1u, 4, false);
    if (!ok) S.fail = 1;
    if (ok) {
      const uint32_t base = smem_u32(S.ring[pipe.stage]) + static_cast<uint32_t>(c_beg + lane) * 16u;
      const uint32_t red = smem_u32(S.red);
      const int nv = rr * nmat;  // virtual rows: rr rows of matrix 0, then rr of matrix 1
#pragma unroll 1
      for (int v0 = 0; v0 < nv; v0 += 4) {
        float acc[4][NC];
#pragma unroll
        for (int v = 0; v < 4; ++v)
#pragma unroll
          for (int c = 0; c < NC; ++c) acc[v][c] = 0.f;
#pragma unroll
        for (int i = 0; i < NCH; ++i) {
          if (c_beg + lane + 32 * i < c_end) {
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              if (v0 + v < nv) {
                float wf[EPC];
                unpack16(lds128(base + static_cast<uint32_t>((v0 + v) * rowb) + i * 512u), wf, WT());
#pragma unroll
                for (int c = 0; c < NC; ++c)
#pragma unroll
                  for (int j = 0; j < EPC; ++j) acc[v][c] = fmaf(wf[j], xr[c][i][j], acc[v][c]);
              }
            }
          }
        }
#pragma unroll
        for (int v = 0; v < 4; ++v)
#pragma unroll
          for (int c = 0; c < NC; ++c) acc[v][c] = warp_sum(acc[v][c]);
        if (lane == 0) {
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            if (v0 + v < nv) {
              const int mat = (v0 + v) / rr, rl = t * R + (v0 + v) % rr;
#pragma unroll
              for (int c = 0; c < NC; ++c) sts32f(red + 4u * (((rl * nmat + mat) * NC + c) * Q + q), acc[v][c]);
            }
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.empty[pipe.stage]);
    pipe.advance();
  }
  named_bar(1, kConsumers);

  // ---- epilogue: sum the slices in fixed order, apply the output rule
  if (!S.fail) {
    const int nout = nr * NC;
    for (int idx = tid; idx < nout; idx += kConsumers) {
      const int rl = idx / NC, c = idx % NC;
      float a = 0.f, b = 0.f;
      for (int qq = 0; qq < Q; ++qq) a += S.red[((rl * nmat + 0) * NC + c) * Q + qq];
      if (nmat == 2)
        for (int qq = 0; qq < Q; ++qq) b += S.red[((rl * nmat + 1) * NC + c) * Q + qq];
      float* y = ph.y[c] + r0 + rl;
      if (ph.epi == EPI_STORE) {
        *y = a;
      } else if (ph.epi == EPI_ADD) {
        *y = (idx == tid ? yres : ldcg(y)) + a;
      } else {
        *y = (a / (1.0f + expf(-a))) * b;
      }
    }
  }
  return pipe;
}

// =========================================================================
// GEMV phase, bf16 weights, on the tensor cores (mma.sync m16n8k16, fp32 accumulate):
// D[16 x 8] += W[16 x 16] · X[16 x 8], where the 16 rows of W are 16 weight rows (a 16-row tile,
// ldmatrix.x4 from shared memory) and the columns of X are the activation columns split into bf16
// hi and lo parts (x = hi + lo to ~2^-17 relative; column 2c = hi, 2c + 1 = lo of activation c;
// ldmatrix.x2 of those rows), so each output is Σ_k w·hi + Σ_k w·lo.  Each warp owns every 8th
// 16-wide k step of a tile; the eight warps' partial sums are added in a fixed order.
// =========================================================================

// The k steps of one K tile for a warp, with the step count fixed at compile time so that the loads
// of later steps are issued ahead of the MMAs of earlier ones: steps st = warp + 8 i for i < S,
// with TAIL one more step st = warp + 8 S when it is below nsteps.  Four accumulation chains.
template <int S, bool TAIL>
__device__ __forceinline__ void tile_steps(uint32_t tb, uint32_t a_off, uint32_t b_ld, int warp, int nsteps,
                                           float (&acc)[4][4]) {
#pragma unroll
  for (int i = 0; i < S + (TAIL ? 1 : 0); ++i) {
    const uint32_t st = static_cast<uint32_t>(warp + kConsumerWarps * i);
    if (TAIL && i == S && static_cast<int>(st) >= nsteps) break;
    uint32_t a0, a1, a2, a3, b0, b1;
    ldmatrix_x4(tb + a_off + 32u * st, a0, a1, a2, a3);
    ldmatrix_x2(b_ld + 32u * st, b0, b1);
    mma_bf16_16816(acc[i & 3], a0, a1, a2, a3, b0, b1);
  }
}

template <int NC>
__device__ __noinline__ Pipe gemv_tiles(const CallParams& cp, const Phase& ph, Smem& S, Pipe pipe, float yres,
                                         float rs0 = 1.f, float rs1 = 1.f);

// GEMV prologue for activations of at most GM·1024 elements per column: the columns into registers
// (GM float4 groups per thread), RMSNorm, the bf16 hi/lo split into shared memory; then the tiles.
template <int NC, int GM>
__device__ __noinline__ Pipe gemv_mma(const CallParams& cp, const Phase& ph, Smem& S, Pipe pipe) {
  const Dims& d = cp.d;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int K = ph.K;
  const bool has_norm = ph.normw != nullptr;
  int r0, nr;
  rows_of(ph, blockIdx.x, gridDim.x, r0, nr);
  float yres = 0.f;
  if (ph.epi == EPI_ADD && tid < nr * NC) yres = ld_out(ph, tid % NC, r0 + tid / NC);

  // ---- activation columns into registers: thread tid holds elements 4·(tid + 256 j) .. +3
  static_assert(GM * 4 * kConsumers * NC <= 10240, "activation registers");
  const int ng = K / 4;
  float4 xv[NC][GM];
  float ss[NC];
#pragma unroll
  for (int c = 0; c < NC; ++c) {
    const GemvCol col = ph.col[c];
    const int* vals = static_cast<const int*>(col.p);
    if (col.src == SRC_BUF && col.tag_back > 0) {
      // tagged words written `tag_back` phases ago: every load first, then the (rare) wait
      const unsigned long long* src = static_cast<const unsigned long long*>(col.p);
      const uint32_t want = pipe.tag - static_cast<uint32_t>(col.tag_back);
      const unsigned long long* ptr[2 * GM];
      ulonglong2 w[2 * GM];
      uint32_t miss = 0u;
#pragma unroll
      for (int j = 0; j < GM; ++j) {
        const int g = min(tid + kConsumers * j, ng - 1);
        ptr[2 * j] = src + 4 * g;
        ptr[2 * j + 1] = src + 4 * g + 2;
        w[2 * j] = ld_relaxed_u64x2(ptr[2 * j]);
        w[2 * j + 1] = ld_relaxed_u64x2(ptr[2 * j + 1]);
      }
#pragma unroll
      for (int i = 0; i < 2 * GM; ++i)
        if (!tags_are(w[i], want)) miss |= 1u << i;
      if (miss != 0u) wait_tagged<2 * GM>(cp, S, ptr, want, miss, w);
#pragma unroll
      for (int j = 0; j < GM; ++j) {
        const int g = tid + kConsumers * j;
        xv[c][j] = g < ng ? make_float4(tval(w[2 * j].x), tval(w[2 * j].y), tval(w[2 * j + 1].x), tval(w[2 * j + 1].y))
                          : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    } else if (col.src == SRC_BUF) {
      const float* src = static_cast<const float*>(col.p);
#pragma unroll
      for (int j = 0; j < GM; ++j) {
        const int g = tid + kConsumers * j;
        xv[c][j] = g < ng ? ldcg4(src + 4 * g) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    } else if (col.src == SRC_FEROW) {
      const int code = ldcgi(vals);
      const unsigned char* row = static_cast<const unsigned char*>(cp.FE) + static_cast<size_t>(code) * K * 2;
#pragma unroll
      for (int j = 0; j < GM; ++j) {
        const int g = tid + kConsumers * j;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (g < ng) {
          const uint2 u = __ldg(reinterpret_cast<const uint2*>(row + static_cast<size_t>(g) * 8));
          v = make_float4(bf16lo(u.x), bf16hi(u.x), bf16lo(u.y), bf16hi(u.y));
        }
        xv[c][j] = v;
      }
    } else {
      // x = sem_scale·E[r0] + m·Σ_cb CE[cb·CBS + code_cb]   (ch.02 §3.2)
      const int tok = ldcgi(vals);
      const float msem = (tok >= d.sem_lo && tok <= d.sem_hi) ? 1.f : 0.f;
#pragma unroll
      for (int j = 0; j < GM; ++j) {
        const int g = tid + kConsumers * j;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (g < ng) {
          const int e = 4 * g;
          float acc[4] = {0.f, 0.f, 0.f, 0.f};
          for (int cb = 0; cb < d.ncb; ++cb) {
            const size_t row = static_cast<size_t>(cb) * d.cbs + ldcgi(vals + 1 + cb);
            const uint2 u = __ldg(reinterpret_cast<const uint2*>(static_cast<const unsigned char*>(cp.CE) + (row * K + e) * 2));
            acc[0] = __fadd_rn(acc[0], bf16lo(u.x));
            acc[1] = __fadd_rn(acc[1], bf16hi(u.x));
            acc[2] = __fadd_rn(acc[2], bf16lo(u.y));
            acc[3] = __fadd_rn(acc[3], bf16hi(u.y));
          }
          const uint2 u = __ldg(reinterpret_cast<const uint2*>(static_cast<const unsigned char*>(cp.E) +
                                                               (static_cast<size_t>(tok) * K + e) * 2));
          v.x = __fadd_rn(__fmul_rn(d.sem_scale, bf16lo(u.x)), __fmul_rn(msem, acc[0]));
          v.y = __fadd_rn(__fmul_rn(d.sem_scale, bf16hi(u.x)), __fmul_rn(msem, acc[1]));
          v.z = __fadd_rn(__fmul_rn(d.sem_scale, bf16lo(u.y)), __fmul_rn(msem, acc[2]));
          v.w = __fadd_rn(__fmul_rn(d.sem_scale, bf16hi(u.y)), __fmul_rn(msem, acc[3]));
        }
        xv[c][j] = v;
      }
    }
    ss[c] = 0.f;
#pragma unroll
    for (int j = 0; j < GM; ++j) {
      const float4 v = xv[c][j];
      ss[c] += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
    }
  }
  if (blockIdx.x == 0) {
    // the raw column written back to its residual row (tagged words with this phase's tag)
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      unsigned long long* wb = reinterpret_cast<unsigned long long*>(ph.col[c].wb);
      if (wb == nullptr) continue;
#pragma unroll
      for (int j = 0; j < GM; ++j) {
        const int g = tid + kConsumers * j;
        if (g < ng) {
          const float4 v = xv[c][j];
          *reinterpret_cast<ulonglong2*>(wb + 4 * g) =
              make_ulonglong2(tagw(__float_as_uint(v.x), pipe.tag), tagw(__float_as_uint(v.y), pipe.tag));
          *reinterpret_cast<ulonglong2*>(wb + 4 * g + 2) =
              make_ulonglong2(tagw(__float_as_uint(v.z), pipe.tag), tagw(__float_as_uint(v.w), pipe.tag));
        }
      }
    }
  }
  // ---- RMSNorm in fp32, with the scale applied after the projection: the activation is multiplied
  // by the norm weight and split at once, the sum of squares is reduced meanwhile, and
  // W·(x·r·w) = r·(W·(x·w)) takes r = 1/sqrt(mean(x²) + eps) in the epilogue
  if (has_norm) {
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      const float t = warp_sum(ss[c]);
      if (lane == 0) S.misc[kMiscSS + warp * NC + c] = t;
    }
    const bool ok = wait_bar(cp, S, &S.full[pipe.stage], pipe.round & 1u, 5, false);
    if (!ok) S.fail = 1;
    const uint32_t nws = smem_u32(S.ring[pipe.stage]);
#pragma unroll
    for (int j = 0; j < GM; ++j) {
      const int g = tid + kConsumers * j;
      if (g < ng) {
        const uint32_t w01 = lds32(nws + 8u * g), w23 = lds32(nws + 8u * g + 4u);
#pragma unroll
        for (int c = 0; c < NC; ++c) {
          float4& v = xv[c][j];
          v.x *= bf16lo(w01);
          v.y *= bf16hi(w01);
          v.z *= bf16lo(w23);
          v.w *= bf16hi(w23);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.empty[pipe.stage]);
    pipe.advance();
  }
  // ---- split into bf16 hi and lo rows: xs row 2c = hi, row 2c+1 = lo (rows padded by 16 bytes so
  // the rows of one ldmatrix sit in different banks)
  const uint32_t xsb = smem_u32(S.xs);
  const uint32_t xpitch = 2u * static_cast<uint32_t>(K) + kTileRowPad;
#pragma unroll
  for (int c = 0; c < NC; ++c) {
#pragma unroll
    for (int j = 0; j < GM; ++j) {
      const int g = tid + kConsumers * j;
      if (g < ng) {
        const float4 v = xv[c][j];
        // packed conversions: hi = bf16(v), lo = bf16(v - hi)
        const uint32_t hi01 = cvt_bf16x2(v.x, v.y), hi23 = cvt_bf16x2(v.z, v.w);
        const float h0 = bf16lo(hi01), h1 = bf16hi(hi01), h2 = bf16lo(hi23), h3 = bf16hi(hi23);
        const uint32_t lo01 = cvt_bf16x2(v.x - h0, v.y - h1), lo23 = cvt_bf16x2(v.z - h2, v.w - h3);
        const uint32_t ahi = xsb + static_cast<uint32_t>(2 * c) * xpitch + 8u * static_cast<uint32_t>(g);
        const uint32_t alo = ahi + xpitch;
        asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(ahi), "r"(hi01), "r"(hi23) : "memory");
        asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(alo), "r"(lo01), "r"(lo23) : "memory");
      }
    }
  }
  named_bar(1, kConsumers);
  float rs[2] = {1.f, 1.f};
  if (has_norm) {
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      float tot = 0.f;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) tot += S.misc[kMiscSS + w * NC + c];
      rs[c] = 1.0f / sqrtf(tot / static_cast<float>(K) + d.eps);
    }
    if (blockIdx.x == 0 && ph.hid_out != nullptr) {
#pragma unroll
      for (int j = 0; j < GM; ++j) {
        const int g = tid + kConsumers * j;
        if (g < ng) {
          const float4 v = xv[0][j];
          *reinterpret_cast<float4*>(ph.hid_out + 4 * g) = make_float4(v.x * rs[0], v.y * rs[0], v.z * rs[0], v.w * rs[0]);
        }
      }
    }
  }

  return gemv_tiles<NC>(cp, ph, S, pipe, yres, rs[0], rs[1]);
}

template <int NC>
__device__ __noinline__ Pipe gemv_tiles(const CallParams& cp, const Phase& ph, Smem& S, Pipe pipe, float yres,
                                         float rs0, float rs1) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int K = ph.K;
  int r0, nr;
  rows_of(ph, blockIdx.x, gridDim.x, r0, nr);
  const uint32_t xsb = smem_u32(S.xs);
  const uint32_t xpitch = 2u * static_cast<uint32_t>(K) + kTileRowPad;
  // ---- tiles: 16-row blocks, each matrix, each K tile; D accumulates over the K tiles.
  const int nmat = ph.nmat;
  // ldmatrix.x2 row addresses for B (lanes 0-15): column n = lane & 7 reads activation row n
  // (2c = hi, 2c + 1 = lo of column c; columns >= 2·NC repeat live rows, their outputs are
  // discarded); matrix 0 = k 0-7 of a step, matrix 1 = k 8-15
  const uint32_t b_ld = order_after(xsb) + static_cast<uint32_t>((lane & 7) % (2 * NC)) * xpitch +
                        static_cast<uint32_t>((lane >> 3) & 1) * 16u;
  const uint32_t red = smem_u32(S.red);
  const int P = nr * ph.nmat * NC;  // partials per warp: [warp][row, matrix, column], conflict-free sums
  const int g = lane >> 2, t = lane & 3;  // D fragment: rows g and g + 8, columns 2t and 2t + 1
  for (int b = 0; b < nr; b += kTileRows) {
    const int rows = min(kTileRows, nr - b);
    // the phase's K tiling (no division per block); a short last block whose rows fit one stage
    // whole takes all of K in one tile (the producer makes the same choice)
    int Kt = ph.Kt, nkt = ph.nkt;
    if (rows < kTileRows && rows * (2 * K + kTileRowPad) <= kStageBytes) {
      Kt = K;
      nkt = 1;
    }
    const uint32_t pitch = static_cast<uint32_t>(Kt) * 2u + kTileRowPad;
    const int nsteps = Kt >> 4;
    // ldmatrix.x4 rows for A: matrices (rows 0-7, k 0-7), (rows 8-15, k 0-7), (rows 0-7, k 8-15),
    // (rows 8-15, k 8-15); rows past the block's last one repeat it (their outputs are discarded)
    const uint32_t a_off = static_cast<uint32_t>(min((lane & 7) + 8 * ((lane >> 3) & 1), rows - 1)) * pitch +
                           static_cast<uint32_t>(lane >> 4) * 16u;
    for (int m = 0; m < nmat; ++m) {
      if (rows == 1 && nkt == 1) {
        // a one-row last block (the rows of a CTA are 16·n + 1): CUDA-core dot products over the
        // whole row (an MMA would use one of its 16 rows); each thread takes 8-element chunks
        const bool ok = wait_bar(cp, S, &S.full[pipe.stage], pipe.round & 1u, 4, false);
        if (!ok) S.fail = 1;
        float dv[NC];
#pragma unroll
        for (int c = 0; c < NC; ++c) dv[c] = 0.f;
        if (ok) {
          const uint32_t tb = order_after(smem_u32(S.ring[pipe.stage]));
          const int nch = K >> 3;
#pragma unroll 2
          for (int ch = tid; ch < nch; ch += kConsumers) {
            const uint4 w = lds128(tb + 16u * static_cast<uint32_t>(ch));
#pragma unroll
            for (int c = 0; c < NC; ++c) {
              const uint32_t xa = xsb + static_cast<uint32_t>(2 * c) * xpitch + 16u * static_cast<uint32_t>(ch);
              const uint4 h = lds128(xa), l = lds128(xa + xpitch);
              const uint32_t wq[4] = {w.x, w.y, w.z, w.w}, hq[4] = {h.x, h.y, h.z, h.w}, lq[4] = {l.x, l.y, l.z, l.w};
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                dv[c] = fmaf(bf16lo(wq[q]), bf16lo(hq[q]) + bf16lo(lq[q]), dv[c]);
                dv[c] = fmaf(bf16hi(wq[q]), bf16hi(hq[q]) + bf16hi(lq[q]), dv[c]);
              }
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.empty[pipe.stage]);
        pipe.advance();
#pragma unroll
        for (int c = 0; c < NC; ++c) {
          const float v = warp_sum(dv[c]);
          if (lane == 0) sts32f(red + 4u * (warp * P + (b * nmat + m) * NC + c), v);
        }
        continue;
      }
      float acc[4][4];
#pragma unroll
      for (int q = 0; q < 4; ++q)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[q][j] = 0.f;
      for (int kt = 0; kt < nkt; ++kt) {
        const bool ok = wait_bar(cp, S, &S.full[pipe.stage], pipe.round & 1u, 4, false);
        if (!ok) S.fail = 1;
        if (ok) {
          const uint32_t tb = order_after(smem_u32(S.ring[pipe.stage]));
          const uint32_t bk = b_ld + 2u * static_cast<uint32_t>(kt * Kt);
          // the K tiles of the S2-Pro projections (1280, 1216 and 1024 columns) have fixed step counts
          if (nsteps == 80) {
            tile_steps<10, false>(tb, a_off, bk, warp, nsteps, acc);
          } else if (nsteps == 76) {
            tile_steps<9, true>(tb, a_off, bk, warp, nsteps, acc);
          } else if (nsteps == 64) {
            tile_steps<8, false>(tb, a_off, bk, warp, nsteps, acc);
          } else {
#pragma unroll 1
            for (int st0 = warp; st0 < nsteps; st0 += 4 * kConsumerWarps) {
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const int st = st0 + q * kConsumerWarps;
                if (st < nsteps) {
                  uint32_t a0, a1, a2, a3, b0, b1;
                  ldmatrix_x4(tb + a_off + 32u * st, a0, a1, a2, a3);
                  ldmatrix_x2(bk + 32u * st, b0, b1);
                  mma_bf16_16816(acc[q], a0, a1, a2, a3, b0, b1);
                }
              }
            }
          }
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) hold(acc[q]);
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.empty[pipe.stage]);
        pipe.advance();
      }
      // column pair (2t, 2t + 1) = (hi, lo) of activation column t: rows g and g + 8
      if (t < NC) {
        const float v0 = ((acc[0][0] + acc[1][0]) + (acc[2][0] + acc[3][0])) +
                         ((acc[0][1] + acc[1][1]) + (acc[2][1] + acc[3][1]));
        const float v1 = ((acc[0][2] + acc[1][2]) + (acc[2][2] + acc[3][2])) +
                         ((acc[0][3] + acc[1][3]) + (acc[2][3] + acc[3][3]));
        if (g < rows) sts32f(red + 4u * (warp * P + ((b + g) * nmat + m) * NC + t), v0);
        if (g + 8 < rows) sts32f(red + 4u * (warp * P + ((b + g + 8) * nmat + m) * NC + t), v1);
      }
    }
  }
  named_bar(1, kConsumers);

  // ---- epilogue: add the warps' partials in a fixed order, apply the output rule
  if (!S.fail) {
    const int nout = nr * NC;
    for (int idx = tid; idx < nout; idx += kConsumers) {
      const int rl = idx / NC, c = idx % NC;
      float a = 0.f, bb = 0.f;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) a += S.red[w * P + (rl * nmat + 0) * NC + c];
      if (nmat == 2)
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) bb += S.red[w * P + (rl * nmat + 1) * NC + c];
      // the norm scale of the column (1 without a norm)
      const float rsc = c == 0 ? rs0 : rs1;
      a *= rsc;
      bb *= rsc;
      float v;
      if (ph.epi == EPI_STORE) {
        v = a;
      } else if (ph.epi == EPI_ADD) {
        v = (idx == tid ? yres : ld_out(ph, c, r0 + rl)) + a;
      } else {
        v = (a / (1.0f + expf(-a))) * bb;
      }
      if (ph.tag_out) {
        // tagged words: the value, or the bf16 hi / lo pair of a planes output
        if (ph.y[c] != nullptr)
          reinterpret_cast<unsigned long long*>(ph.y[c])[r0 + rl] = tagw(__float_as_uint(v), pipe.tag);
        if (ph.yp[c] != nullptr) {
          const float hi = bf16lo(cvt_bf16x2(v, 0.f));
          reinterpret_cast<unsigned long long*>(ph.yp[c])[r0 + rl] = tagw(cvt_bf16x2(hi, v - hi), pipe.tag);
        }
      } else {
        if (ph.y[c] != nullptr) ph.y[c][r0 + rl] = v;
        if (ph.yp[c] != nullptr) store_planes(ph.yp[c], ph.M, r0 + rl, v);
      }
    }
  }
  return pipe;
}

// The activation comes as bf16 hi / lo rows written by the producing phase: one bulk copy per row
// into xs, then the tiles (no normalisation on this path).
template <int NC>
__device__ __noinline__ Pipe gemv_planes(const CallParams& cp, const Phase& ph, Smem& S, Pipe pipe) {
  const int tid = threadIdx.x;
  const int K = ph.K;
  int r0, nr;
  rows_of(ph, blockIdx.x, gridDim.x, r0, nr);
  float yres = 0.f;
  if (ph.epi == EPI_ADD && tid < nr * NC) yres = ld_out(ph, tid % NC, r0 + tid / NC);
  const uint32_t xpitch = 2u * static_cast<uint32_t>(K) + kTileRowPad;
  if (ph.col[0].tag_back > 0) {
    // tagged planes words (hi | lo << 16, then the tag), written tag_back phases ago: every load
    // of a thread in flight at once (one round up to K = 9728), unpacked into the hi and lo rows
    // of xs
    constexpr int B = 19;  // element pairs per thread and round: K <= 9728 in one round
    const uint32_t xsb = smem_u32(S.xs);
    const int npairs = K / 2;
#pragma unroll 1
    for (int c = 0; c < NC; ++c) {
      const unsigned long long* src = static_cast<const unsigned long long*>(ph.col[c].p);
      const uint32_t want = pipe.tag - static_cast<uint32_t>(ph.col[c].tag_back);
#pragma unroll 1
      for (int base = tid; base < npairs; base += B * kConsumers) {
        const unsigned long long* ptr[B];
        ulonglong2 w[B];
        uint32_t miss = 0u;
#pragma unroll
        for (int i = 0; i < B; ++i) {
          ptr[i] = src + 2 * min(base + i * kConsumers, npairs - 1);
          w[i] = ld_relaxed_u64x2(ptr[i]);
        }
#pragma unroll
        for (int i = 0; i < B; ++i)
          if (!tags_are(w[i], want)) miss |= 1u << i;
        if (miss != 0u) wait_tagged<B>(cp, S, ptr, want, miss, w);
#pragma unroll
        for (int i = 0; i < B; ++i) {
          const int q = base + i * kConsumers;
          if (q < npairs) {
            const uint32_t e0 = static_cast<uint32_t>(w[i].x), e1 = static_cast<uint32_t>(w[i].y);
            const uint32_t hi2 = (e0 & 0xffffu) | (e1 << 16), lo2 = (e0 >> 16) | (e1 & 0xffff0000u);
            const uint32_t a = xsb + static_cast<uint32_t>(2 * c) * xpitch + 4u * static_cast<uint32_t>(q);
            asm volatile("st.shared.u32 [%0], %1;" ::"r"(a), "r"(hi2) : "memory");
            asm volatile("st.shared.u32 [%0], %1;" ::"r"(a + xpitch), "r"(lo2) : "memory");
          }
        }
      }
    }
    named_bar(1, kConsumers);
    return gemv_tiles<NC>(cp, ph, S, pipe, yres);
  }
  if (tid == 0) {
    // the previous users of xs (generic-proxy accesses, ordered before by the phase barrier) come
    // before these async-proxy writes
    fence_proxy_async_smem();
    const uint32_t rowb = 2u * static_cast<uint32_t>(K);
    mbar_arrive_expect_tx(&S.xsbar, 2u * NC * rowb);
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      const uint16_t* pl = static_cast<const uint16_t*>(ph.col[c].p);
      bulk_g2s_plain(S.xs + (2 * c) * xpitch, pl, rowb, &S.xsbar);
      bulk_g2s_plain(S.xs + (2 * c + 1) * xpitch, pl + K, rowb, &S.xsbar);
    }
  }
  const bool ok = wait_bar(cp, S, &S.xsbar, pipe.xs_uses & 1u, 6, false);
  if (!ok) {
    S.fail = 1;
    if (tid == 0) drain_copies(cp, &S.xsbar, pipe.xs_uses & 1u, 7);  // this CTA's own copies
  }
  ++pipe.xs_uses;
  return gemv_tiles<NC>(cp, ph, S, pipe, yres);
}

template <class C>
__device__ __forceinline__ Pipe gemv(const CallParams& cp, const Phase& ph, Smem& S, Pipe pipe) {
  if constexpr (C::bf16) {
    if (ph.col[0].src == SRC_PLANES) {
      return ph.ncols == 1 ? gemv_planes<1>(cp, ph, S, pipe) : gemv_planes<2>(cp, ph, S, pipe);
    }
    // the activation length selects how many float4 groups each thread holds (K <= GM·1024)
    if (ph.ncols == 1) {
      if (ph.K <= 3072) return gemv_mma<1, 3>(cp, ph, S, pipe);
      if (ph.K <= 4096) return gemv_mma<1, 4>(cp, ph, S, pipe);
      return gemv_mma<1, 10>(cp, ph, S, pipe);
    } else {
      if (ph.K <= 3072) return gemv_mma<2, 3>(cp, ph, S, pipe);
      return gemv_mma<2, 5>(cp, ph, S, pipe);
    }
  } else {
    return ph.ncols == 1 ? gemv_t<float, 1>(cp, ph, S, pipe) : gemv_t<float, 2>(cp, ph, S, pipe);
  }
}

// =========================================================================
// per-head RMSNorm + RoPE of one head vector held by a warp (lane holds DPL contiguous values)
// =========================================================================

// the head's norm weights and RoPE row held by a lane (loaded before the head vector itself, so
// that their loads overlap it)
template <int DPL>
struct NormRope {
  float w[DPL];
  float2 cs[DPL / 2];
};

template <int DPL>
__device__ __forceinline__ void load_norm_rope(NormRope<DPL>& nr, const void* nw, int esz, bool norm,
                                               const float2* rope_row) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int j = 0; j < DPL; ++j) nr.w[j] = norm ? wload(nw, lane * DPL + j, esz) : 1.f;
#pragma unroll
  for (int j = 0; j < DPL; j += 2) nr.cs[j >> 1] = rope_row[(lane * DPL + j) >> 1];
}

template <int DPL>
__device__ __forceinline__ void head_norm_rope(float (&v)[DPL], const NormRope<DPL>& nr, float eps, int hd, bool norm) {
  if (norm) {
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < DPL; ++j) s += v[j] * v[j];
    s = warp_sum(s);
    const float r = 1.0f / sqrtf(s / static_cast<float>(hd) + eps);
#pragma unroll
    for (int j = 0; j < DPL; ++j) v[j] = (v[j] * r) * nr.w[j];
  }
#pragma unroll
  for (int j = 0; j < DPL; j += 2) {
    const float2 cs = nr.cs[j >> 1];
    const float a = v[j], b = v[j + 1];
    v[j] = a * cs.x - b * cs.y;
    v[j + 1] = a * cs.y + b * cs.x;
  }
}

// per-head RMSNorm + RoPE of one head vector held by a warp (lane holds DPL contiguous values)
template <int DPL>
__device__ __forceinline__ void head_norm_rope(float (&v)[DPL], const void* nw, int esz, float eps, int hd,
                                               bool norm, const float2* rope_row) {
  NormRope<DPL> nr;
  load_norm_rope<DPL>(nr, nw, esz, norm, rope_row);
  head_norm_rope<DPL>(v, nr, eps, hd, norm);
}

template <typename KT>
__device__ __forceinline__ float kv_to_f(KT x);
template <>
__device__ __forceinline__ float kv_to_f<__half>(__half x) { return __half2float(x); }
template <>
__device__ __forceinline__ float kv_to_f<float>(float x) { return x; }
template <typename KT>
__device__ __forceinline__ KT f_to_kv(float x);
template <>
__device__ __forceinline__ __half f_to_kv<__half>(float x) { return __float2half_rn(x); }
template <>
__device__ __forceinline__ float f_to_kv<float>(float x) { return x; }

// four consecutive elements of a K/V row in shared memory (8- or 16-byte aligned) to fp32
template <typename KT>
__device__ __forceinline__ void load4_kv(const KT* p, float (&f)[4]) {
  if constexpr (sizeof(KT) == 2) {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
    const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
    f[0] = a.x;
    f[1] = a.y;
    f[2] = b.x;
    f[3] = b.y;
  } else {
    const float4 u = *reinterpret_cast<const float4*>(p);
    f[0] = u.x;
    f[1] = u.y;
    f[2] = u.z;
    f[3] = u.w;
  }
}


// =========================================================================
// Slow-AR attention: q/k norm + RoPE, KV store of the new slot, split-K decode attention over
// slots 0..pos.  Item = (KV head, split); each writes its unnormalised output with its running
// max and denominator, and the last split of a KV head to finish combines them.
// Rounds of RS slots: the K and V rows of the next round are copied into shared memory
// (cp.async, double-buffered) while the current one is processed.  Scores: TPS threads per slot,
// thread sp taking the 4-element chunks sp, sp + TPS, ... of the row, so that at each step the
// threads of a slot read one contiguous span of q (a broadcast across the warp's slots, free of
// bank conflicts); P·V: each thread owns fixed (head, element) outputs and reads the
// probabilities of 4 slots at once.
// =========================================================================

// The combine of the Slow-AR split partials of KV head g (the last split to arrive): for each of
// its rep heads h and elements e, o = Σ_s e^{m_s - M} o_s / Σ_s e^{m_s - M} l_s over the ns splits
// in split order; (m_s, l_s) of head h at mls[2 (h ns + s)].  NSM bounds ns (the unrolled length).
template <int NSM, int HD>
__device__ __forceinline__ void combine_splits(const CallParams& cp, const Phase& ph, const float* mls, int g, int ns,
                                               int rep) {
  static_assert(4 * HD <= 2 * kConsumers, "combine outputs per thread");
  const int tid = threadIdx.x;
  float pv[2][NSM];
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const int idx = tid + q * kConsumers, r = idx / HD, e = idx % HD;
#pragma unroll
    for (int s2 = 0; s2 < NSM; ++s2)
      pv[q][s2] = (idx < rep * HD && s2 < ns) ? ldcg(cp.part + (static_cast<size_t>(g * ns + s2) * 4 + r) * HD + e) : 0.f;
  }
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const int idx = tid + q * kConsumers, r = idx / HD, e = idx % HD;
    if (idx >= rep * HD) continue;
    const float* mr = mls + 2 * r * ns;
    float M = -INFINITY;
#pragma unroll
    for (int s2 = 0; s2 < NSM; ++s2)
      if (s2 < ns) M = fmaxf(M, mr[2 * s2]);
    float o = 0.f, l = 0.f;
#pragma unroll
    for (int s2 = 0; s2 < NSM; ++s2) {
      if (s2 < ns) {
        const float w = expf(mr[2 * s2] - M);
        o += w * pv[q][s2];
        l += w * mr[2 * s2 + 1];
      }
    }
    ph.out[(g * rep + r) * HD + e] = o / l;
    if (ph.outp != nullptr) store_planes(ph.outp, cp.d.Hq * HD, (g * rep + r) * HD + e, o / l);
  }
}

template <typename KT, int HD>
__device__ __noinline__ void attn_slow_t(const CallParams& cp, const Phase& ph, Smem& S, uint32_t tag) {
  constexpr int RB = HD * static_cast<int>(sizeof(KT));  // bytes per K/V row
  constexpr int RS = kXsStageBytes / RB;                 // slots per round (16, 32 or 64)
  constexpr int TPS = kConsumers / RS;                   // threads per slot in the scores
  constexpr int EPS = HD / TPS;                          // elements per thread in the scores
  constexpr int CPS = RB / 16;                           // 16-byte chunks per row
  constexpr int OPT = 4 * HD / kConsumers;               // outputs per thread in P·V
  constexpr int DPL = HD / 32;
  static_assert(RS <= 64 && EPS * static_cast<int>(sizeof(KT)) == 32 && EPS % 4 == 0, "attention round layout");
  const Dims& d = cp.d;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rep = S.attn_rep;
  const int pos = S.pos_frame;
  const int n = pos + 1;
  const int G = gridDim.x;
  const int ns = S.attn_ns, chunk = S.attn_chunk;
  const int nitems = d.Hkv * ns;
  const float sc_mul = ph.scale;  // 1/sqrt(head_dim)
  const size_t kvh = static_cast<size_t>(cp.kv_slots) * HD;  // elements per KV head
  const KT* Kc = static_cast<const KT*>(ph.kc);
  const KT* Vc = static_cast<const KT*>(ph.vc);
  const float2* rope_row = cp.rope + static_cast<size_t>(pos) * (HD / 2);
  KT* kst = reinterpret_cast<KT*>(S.xs);                        // [2][RS][HD]
  KT* vst = reinterpret_cast<KT*>(S.xs + 2 * kXsStageBytes);    // [2][RS][HD]
  float* xsf = reinterpret_cast<float*>(S.xs);
  float* qs = xsf + kXsQ;
  float* knew = xsf + kXsKV;
  float* vnew = xsf + kXsKV + 128;
  float* ps = xsf + kXsSc;
  float* stat = xsf + kXsStat;
  float* pml = const_cast<float*>(S.attn_pml);
  const int ss = tid / TPS, sp = tid % TPS;  // scores: slot, part
  const int oe = tid % HD, oh = tid / HD;    // P·V: element, first head (then + kConsumers / HD)

  for (int item = blockIdx.x; item < nitems; item += G) {
    const bool own = item == static_cast<int>(blockIdx.x);  // the item planned at the frame start
    const int g = own ? S.attn_g : item / ns, s = own ? S.attn_s : item % ns;
    const int j0 = s * chunk, j1 = min(n, j0 + chunk);
    const bool has_new = (j1 == n);
    const int nrounds = (j1 - j0 + RS - 1) / RS;
    const KT* Kg = Kc + g * kvh;
    const KT* Vg = Vc + g * kvh;
    // K and V rows of round r into buffer r & 1 (the new slot is filled from shared memory)
    auto issue = [&](int r) {
      const int b0 = j0 + r * RS;
      for (int i = tid; i < RS * CPS; i += kConsumers) {
        const int sl = i / CPS, ch = i % CPS, slot = b0 + sl;
        if (slot < j1 && slot != pos) {
          const size_t off = static_cast<size_t>(slot) * HD + ch * (16 / sizeof(KT));
          const size_t so = (static_cast<size_t>(r & 1) * RS + sl) * HD + ch * (16 / sizeof(KT));
          cp_async16(kst + so, Kg + off);
          cp_async16(vst + so, Vg + off);
        }
      }
      cp_async_commit();
    };
    issue(0);
    // ---- q heads of this KV head; the new slot's k (normed, rotated) and v, stored in the cache
    if (warp < rep) {
      const int h = g * rep + warp;
      NormRope<DPL> nr;
      load_norm_rope<DPL>(nr, ph.qn, d.esz, d.qk_norm != 0, rope_row);
      float v[DPL];
      QkvWords<DPL> tq;
      qkv_issue<DPL>(ph, static_cast<size_t>(h) * HD + lane * DPL, tq, v);
      qkv_ready<DPL>(cp, S, ph, tag, tq, v);
      head_norm_rope<DPL>(v, nr, d.eps, HD, d.qk_norm != 0);
#pragma unroll
      for (int j = 0; j < DPL; ++j) qs[warp * HD + lane * DPL + j] = v[j];
    } else if (warp == rep && has_new) {
      NormRope<DPL> nr;
      load_norm_rope<DPL>(nr, ph.kn, d.esz, d.qk_norm != 0, rope_row);
      float k[DPL], v[DPL];
      QkvWords<DPL> tk, tv;
      qkv_issue<DPL>(ph, static_cast<size_t>(d.Hq + g) * HD + lane * DPL, tk, k);
      qkv_issue<DPL>(ph, static_cast<size_t>(d.Hq + d.Hkv + g) * HD + lane * DPL, tv, v);
      qkv_ready<DPL>(cp, S, ph, tag, tk, k);
      qkv_ready<DPL>(cp, S, ph, tag, tv, v);
      head_norm_rope<DPL>(k, nr, d.eps, HD, d.qk_norm != 0);
      KT* kd = const_cast<KT*>(Kc) + g * kvh + static_cast<size_t>(pos) * HD + lane * DPL;
      KT* vd = const_cast<KT*>(Vc) + g * kvh + static_cast<size_t>(pos) * HD + lane * DPL;
#pragma unroll
      for (int j = 0; j < DPL; ++j) {
        const KT kq = f_to_kv<KT>(k[j]), vq = f_to_kv<KT>(v[j]);
        kd[j] = kq;
        vd[j] = vq;
        knew[lane * DPL + j] = kv_to_f<KT>(kq);
        vnew[lane * DPL + j] = kv_to_f<KT>(vq);
      }
    }
    float acc[OPT];
#pragma unroll
    for (int j = 0; j < OPT; ++j) acc[j] = 0.f;
    float m_run = -INFINITY, l_run = 0.f;  // warps r < rep
#pragma unroll 1
    for (int r = 0; r < nrounds; ++r) {
      named_bar(1, kConsumers);  // round r - 1 is fully consumed: its buffer may be refilled
      if (r + 1 < nrounds) {
        issue(r + 1);
        cp_async_wait_group<1>();
      } else {
        cp_async_wait_group<0>();
      }
      const int b0 = j0 + r * RS, L = min(RS, j1 - b0);
      const int buf = r & 1;
      if (pos >= b0 && pos < b0 + L && tid < HD) {
        const size_t so = (static_cast<size_t>(buf) * RS + (pos - b0)) * HD + tid;
        kst[so] = f_to_kv<KT>(knew[tid]);
        vst[so] = f_to_kv<KT>(vnew[tid]);
      }
      named_bar(1, kConsumers);
      // ---- scores: slot ss, chunks sp + c·TPS (4 elements each) of each of the rep q heads
      {
        const KT* kr = kst + (static_cast<size_t>(buf) * RS + ss) * HD;
        float dot[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int c = 0; c < EPS / 4; ++c) {
          const int e0 = (c * TPS + sp) * 4;
          float kf[4];
          load4_kv<KT>(kr + e0, kf);
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            if (h < rep) {
              const float4 q = *reinterpret_cast<const float4*>(qs + h * HD + e0);
              dot[h] = fmaf(q.x, kf[0], dot[h]);
              dot[h] = fmaf(q.y, kf[1], dot[h]);
              dot[h] = fmaf(q.z, kf[2], dot[h]);
              dot[h] = fmaf(q.w, kf[3], dot[h]);
            }
          }
        }
#pragma unroll
        for (int off = TPS / 2; off >= 1; off >>= 1)
#pragma unroll
          for (int h = 0; h < 4; ++h) dot[h] += __shfl_xor_sync(0xffffffffu, dot[h], off);
        if (sp == 0)
#pragma unroll
          for (int h = 0; h < 4; ++h)
            if (h < rep) ps[h * 64 + ss] = ss < L ? dot[h] * sc_mul : -INFINITY;
      }
      named_bar(1, kConsumers);
      // ---- online softmax of the round (warp h: head h)
      if (warp < rep) {
        float* row = ps + warp * 64;
        const float v0 = lane < RS ? row[lane] : -INFINITY;
        const float v1 = lane + 32 < RS ? row[lane + 32] : -INFINITY;
        const float mnew = fmaxf(m_run, warp_max(fmaxf(v0, v1)));
        const float alpha = expf(m_run - mnew);
        const float p0 = expf(v0 - mnew), p1 = expf(v1 - mnew);
        if (lane < RS) row[lane] = p0;
        if (lane + 32 < RS) row[lane + 32] = p1;
        l_run = l_run * alpha + warp_sum(p0 + p1);
        m_run = mnew;
        if (lane == 0) stat[warp] = alpha;
      }
      named_bar(1, kConsumers);
      // ---- P·V: outputs (head oh + j·(kConsumers / HD), element oe)
#pragma unroll
      for (int j = 0; j < OPT; ++j) {
        const int h = oh + j * (kConsumers / HD);
        acc[j] *= h < rep ? stat[h] : 0.f;
      }
      const KT* vr = vst + static_cast<size_t>(buf) * RS * HD + oe;
      const int L4 = L & ~3;
#pragma unroll 2
      for (int sl = 0; sl < L4; sl += 4) {
        float v[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) v[t] = kv_to_f<KT>(vr[static_cast<size_t>(sl + t) * HD]);
#pragma unroll
        for (int j = 0; j < OPT; ++j) {
          const int h = oh + j * (kConsumers / HD);
          if (h < rep) {
            const float4 p = *reinterpret_cast<const float4*>(ps + h * 64 + sl);
            acc[j] = fmaf(p.x, v[0], acc[j]);
            acc[j] = fmaf(p.y, v[1], acc[j]);
            acc[j] = fmaf(p.z, v[2], acc[j]);
            acc[j] = fmaf(p.w, v[3], acc[j]);
          }
        }
      }
      for (int sl = L4; sl < L; ++sl) {
        const float v = kv_to_f<KT>(vr[static_cast<size_t>(sl) * HD]);
#pragma unroll
        for (int j = 0; j < OPT; ++j) {
          const int h = oh + j * (kConsumers / HD);
          if (h < rep) acc[j] = fmaf(ps[h * 64 + sl], v, acc[j]);
        }
      }
    }
    if (warp < rep && lane == 0) {
      stat[4 + warp] = m_run;
      stat[8 + warp] = l_run;
    }
    named_bar(1, kConsumers);
#pragma unroll
    for (int j = 0; j < OPT; ++j) {
      const int h = oh + j * (kConsumers / HD);
      if (h < rep) {
        if (ns == 1) {
          const float o = acc[j] / stat[8 + h];
          ph.out[(g * rep + h) * HD + oe] = o;
          if (ph.outp != nullptr) store_planes(ph.outp, d.Hq * HD, (g * rep + h) * HD + oe, o);
        } else {
          cp.part[(static_cast<size_t>(item) * 4 + h) * HD + oe] = acc[j];
        }
      }
    }
    if (ns == 1) {
      named_bar(1, kConsumers);
      continue;
    }
    if (tid < rep) {
      pml[(static_cast<size_t>(item) * 4 + tid) * 2] = stat[4 + tid];
      pml[(static_cast<size_t>(item) * 4 + tid) * 2 + 1] = stat[8 + tid];
    }
    // ---- the last split of this KV head to arrive combines all of them:
    //   o = Σ_s e^{m_s - M} o_s / Σ_s e^{m_s - M} l_s
    // The CTA's partials are ordered before thread 0's ticket by the barrier; the ticket is a
    // release (publishing them) and an acquire (the last arriver sees every split's partials).
    named_bar(1, kConsumers);
    if (tid == 0) {
      const unsigned t = atom_add_acq_rel_gpu(&cp.ctl->tickets[g], 1u);
      S.flag = (t == static_cast<unsigned>(ns - 1)) ? 1 : 0;
      if (S.flag) cp.ctl->tickets[g] = 0u;  // every split of this item has arrived
    }
    named_bar(1, kConsumers);
    if (S.flag) {
      float* mls = stat + 16;
#pragma unroll 1
      for (int i = tid; i < rep * ns; i += kConsumers) {
        const int r = i / ns, s2 = i % ns;
        const float2 ml = __ldcg(reinterpret_cast<const float2*>(pml + (static_cast<size_t>(g * ns + s2) * 4 + r) * 2));
        mls[2 * i] = ml.x;
        mls[2 * i + 1] = ml.y;
      }
      named_bar(1, kConsumers);
      // at most 4 heads x 128 elements: two outputs per thread, every split's partial of both
      // requested at once (the sums keep split order); the unrolled length follows ns
      if (ns <= 8) combine_splits<8, HD>(cp, ph, mls, g, ns, rep);
      else if (ns <= 16) combine_splits<16, HD>(cp, ph, mls, g, ns, rep);
      else combine_splits<kAttnMaxSplits, HD>(cp, ph, mls, g, ns, rep);
    }
    named_bar(1, kConsumers);
  }
}

template <class C>
__device__ void attn_slow(const CallParams& cp, const Phase& ph, Smem& S, uint32_t tag) {
  attn_slow_t<typename C::KT, C::hd>(cp, ph, S, tag);
}

// =========================================================================
// Fast-AR attention over the frame's window (positions 0..pos0+npos-1), causal offset 0.
// One warp per (new position, query head); the within-frame K/V (fp32) of earlier positions
// come from the window cache, the new ones are recomputed by each warp that needs them.
// =========================================================================

template <int HD>
__device__ __noinline__ void attn_fast_t(const CallParams& cp, const Phase& ph, Smem& S, uint32_t tag) {
  // One CTA per (position, query head); its eight warps split the window's slots (warp w: slots
  // w and w + 8), so each warp issues its few key / value loads at once instead of walking the
  // slots one dependent load after another.  Each warp keeps an online-softmax partial (max,
  // sum, weighted values); warp 0 combines the eight in warp order.
  constexpr int DPL = HD / 32;
  constexpr int kSlotsPerWarp = 2;  // window <= 16 positions
  const Dims& d = cp.d;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int H = d.Hqf, Hk = d.Hkvf, rep = S.fa_rep;
  const int QKV = (H + 2 * Hk) * HD;
  const int nitems = ph.npos * H;
  const float sc_mul = ph.scale;
  float* kc = static_cast<float*>(ph.kc);  // [Wf][Hk][HD]
  float* vc = static_cast<float*>(ph.vc);
  float* part = reinterpret_cast<float*>(S.xs);  // per warp: o[HD], max, sum
  for (int item = blockIdx.x; item < nitems; item += gridDim.x) {
    const bool own = item == static_cast<int>(blockIdx.x);  // the item planned at the launch start
    const int jn = own ? S.fa_j : item / H, h = own ? S.fa_h : item % H, g = own ? S.fa_g : h / rep;
    const int p = ph.pos0 + jn;
    // every load first: the query, and the keys / values of this warp's slots (the frame's new
    // positions from the projection output, earlier ones from the window cache)
    NormRope<DPL> nq;
    load_norm_rope<DPL>(nq, ph.qn, d.esz, d.qk_norm != 0, cp.rope_f + static_cast<size_t>(p) * (HD / 2));
    float q[DPL];
    QkvWords<DPL> tq, tk[kSlotsPerWarp], tv[kSlotsPerWarp];
    qkv_issue<DPL>(ph, static_cast<size_t>(jn) * QKV + h * HD + lane * DPL, tq, q);
    float k[kSlotsPerWarp][DPL], v[kSlotsPerWarp][DPL];
    NormRope<DPL> nk[kSlotsPerWarp];
#pragma unroll
    for (int t = 0; t < kSlotsPerWarp; ++t) {
      const int s = warp + kConsumerWarps * t;
      if (s > p) continue;  // uniform across the warp
      if (s >= ph.pos0) {
        load_norm_rope<DPL>(nk[t], ph.kn, d.esz, d.qk_norm != 0, cp.rope_f + static_cast<size_t>(s) * (HD / 2));
        const size_t row = static_cast<size_t>(s - ph.pos0) * QKV;
        qkv_issue<DPL>(ph, row + (H + g) * HD + lane * DPL, tk[t], k[t]);
        qkv_issue<DPL>(ph, row + (H + Hk + g) * HD + lane * DPL, tv[t], v[t]);
      } else {
        const size_t off = (static_cast<size_t>(s) * Hk + g) * HD + lane * DPL;
#pragma unroll
        for (int j = 0; j < DPL; ++j) {
          k[t][j] = ldcg(kc + off + j);
          v[t][j] = ldcg(vc + off + j);
        }
      }
    }
    qkv_ready<DPL>(cp, S, ph, tag, tq, q);
    head_norm_rope<DPL>(q, nq, d.eps, HD, d.qk_norm != 0);
    float m = -INFINITY, sc[kSlotsPerWarp];
#pragma unroll
    for (int t = 0; t < kSlotsPerWarp; ++t) {
      const int s = warp + kConsumerWarps * t;
      sc[t] = -INFINITY;
      if (s > p) continue;  // uniform across the warp
      if (s >= ph.pos0) {
        // a new position of this frame: its key is normalised and rotated here
        qkv_ready<DPL>(cp, S, ph, tag, tk[t], k[t]);
        qkv_ready<DPL>(cp, S, ph, tag, tv[t], v[t]);
        head_norm_rope<DPL>(k[t], nk[t], d.eps, HD, d.qk_norm != 0);
        if (s == p && (h % rep) == 0) {
#pragma unroll
          for (int j = 0; j < DPL; ++j) {
            kc[(static_cast<size_t>(s) * Hk + g) * HD + lane * DPL + j] = k[t][j];
            vc[(static_cast<size_t>(s) * Hk + g) * HD + lane * DPL + j] = v[t][j];
          }
        }
      }
      float dot = 0.f;
#pragma unroll
      for (int j = 0; j < DPL; ++j) dot += q[j] * k[t][j];
      sc[t] = warp_sum(dot) * sc_mul;
      m = fmaxf(m, sc[t]);
    }
    float l = 0.f, o[DPL];
#pragma unroll
    for (int j = 0; j < DPL; ++j) o[j] = 0.f;
#pragma unroll
    for (int t = 0; t < kSlotsPerWarp; ++t) {
      if (sc[t] == -INFINITY) continue;
      const float e = expf(sc[t] - m);
      l += e;
#pragma unroll
      for (int j = 0; j < DPL; ++j) o[j] += e * v[t][j];
    }
    float* pw = part + warp * (HD + 2);
#pragma unroll
    for (int j = 0; j < DPL; ++j) pw[lane * DPL + j] = o[j];
    if (lane == 0) {
      pw[HD] = m;
      pw[HD + 1] = l;
    }
    named_bar(1, kConsumers);
    if (warp == 0) {
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, part[w * (HD + 2) + HD]);
      float L = 0.f, O[DPL];
#pragma unroll
      for (int j = 0; j < DPL; ++j) O[j] = 0.f;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) {
        const float mw = part[w * (HD + 2) + HD];
        if (mw == -INFINITY) continue;  // a warp without slots
        const float f = expf(mw - M);
        L += part[w * (HD + 2) + HD + 1] * f;
#pragma unroll
        for (int j = 0; j < DPL; ++j) O[j] += part[w * (HD + 2) + lane * DPL + j] * f;
      }
#pragma unroll
      for (int j = 0; j < DPL; ++j) {
        const float ov = O[j] / L;
        ph.out[static_cast<size_t>(jn) * (H * HD) + h * HD + lane * DPL + j] = ov;
        if (ph.outp != nullptr)
          store_planes(ph.outp + static_cast<size_t>(jn) * 2 * (H * HD), H * HD, h * HD + lane * DPL + j, ov);
      }
    }
    named_bar(1, kConsumers);  // the partials are read before the next item overwrites them
  }
}

template <class C>
__device__ void attn_fast(const CallParams& cp, const Phase& ph, Smem& S, uint32_t tag) {
  attn_fast_t<C::hd>(cp, ph, S, tag);
}

// caller-supplied ids (forced draws, Fast-AR-alone prefixes) are checked before any use as an index
__device__ __forceinline__ int checked_id(const CallParams& cp, int v, int hi) {
  if (v < 0 || v >= hi) {
    atomicCAS(&cp.ctl->error, 0, S2_EINVAL);
    return 0;
  }
  return v;
}

__device__ void copy_vec(float* dst, const float* src, int n) {
  for (int i = threadIdx.x; i < n; i += kConsumers) dst[i] = ldcg(src + i);
}

// main draw, repetition-aware redraw, clamp, stop (CTA 0)
__device__ __noinline__ void sample_main(const CallParams& cp, Smem& S, int f) {
  const Dims& d = cp.d;
  StreamState* st = cp.st;
  const int fd = ldcgi(&st->frames_done);
  if (cp.dbg_main) copy_vec(cp.dbg_main + static_cast<size_t>(f) * d.A, cp.logits, d.A);
  if (cp.dbg_hidden) copy_vec(cp.dbg_hidden + static_cast<size_t>(f) * d.D, cp.hidden, d.D);
  const float* E = cp.expo + static_cast<size_t>(f) * kDraws * kTopK;
  const bool block_end = fd < cp.min_tokens;
  // a stop request (s2_stop_stream) ends the stream at this frame boundary, like im_end
  if (threadIdx.x == 0) S.flag = ld_volatile_int(&st->stop_req);
  named_bar(1, kConsumers);
  const int stop = S.flag;
  named_bar(1, kConsumers);
  if (stop) {
    if (threadIdx.x == 0) {
      st->done = 1;
      st->n_out = f;
    }
    return;
  }
  int d0 = draw(cp.d, *reinterpret_cast<SampScratch*>(S.xs), cp.logits, d.A, true, block_end, cp.temperature, cp.top_p, E);
  if (threadIdx.x == 0) {
    if (cp.dbg_draws) cp.dbg_draws[f * kDraws + 0] = d0;
    if (cp.forced) {
      d0 = cp.forced[f * kDraws + 0];
      if (d0 < 0 || d0 >= d.V) {
        atomicCAS(&cp.ctl->error, 0, S2_EINVAL);
        d0 = d.im_end;  // an invalid forced token ends the stream
      }
    }
    S.flag = d0;
  }
  named_bar(1, kConsumers);
  d0 = S.flag;
  named_bar(1, kConsumers);
  if (d0 == d.im_end || d0 < 0) {
    if (threadIdx.x == 0) {
      st->done = 1;
      st->n_out = f;
      if (cp.dbg_draws)
        for (int k = 1; k < kDraws; ++k) cp.dbg_draws[f * kDraws + k] = -1;
    }
    return;
  }
  int d1 = draw(cp.d, *reinterpret_cast<SampScratch*>(S.xs), cp.logits, d.A, true, block_end, cp.ras_temperature, cp.ras_top_p, E + kTopK);
  if (threadIdx.x < 32) {
    // warp 0: the RAS window is read, tested and shifted by its lanes at once (lane i: entry i)
    const int lane = threadIdx.x;
    if (lane == 0) {
      if (cp.dbg_draws) cp.dbg_draws[f * kDraws + 1] = d1;
      if (cp.forced) d1 = checked_id(cp, cp.forced[f * kDraws + 1], d.V);
      if (d1 < 0) d1 = d0;
    }
    d1 = __shfl_sync(0xffffffffu, d1, 0);
    const int wl = ldcgi(&st->wlen);
    const int wv = lane < wl ? ldcgi(&st->window[lane]) : -1;
    const bool seen = __any_sync(0xffffffffu, lane < wl && wv == d0);
    const bool trig = seen && d0 >= d.sem_lo && d0 <= d.sem_hi;
    const int tok = trig ? d1 : d0;
    if (wl < cp.ras_window) {
      if (lane == 0) {
        st->window[wl] = tok;
        st->wlen = wl + 1;
      }
    } else {
      if (lane >= 1 && lane < wl) st->window[lane - 1] = wv;
      if (lane == 0) st->window[wl - 1] = tok;
    }
    if (lane == 0) {
      int code0 = tok - d.sem_lo;
      code0 = code0 < 0 ? 0 : (code0 > d.cbs - 1 ? d.cbs - 1 : code0);
      st->vals[0] = tok;
      st->vals[1] = code0;
      cp.fcode[0] = code0;
      cp.stage[static_cast<size_t>(f) * d.ncb + 0] = code0;
      st->frames_done = fd + 1;
    }
  }
}

// one Fast-AR draw (CTA 0), codebook c = 1..NCB-1
__device__ __noinline__ void sample_fast(const CallParams& cp, Smem& S, int f, int c) {
  const Dims& d = cp.d;
  if (cp.fast_only) {
    copy_vec(cp.fout + (static_cast<size_t>(f) * (d.ncb - 1) + (c - 1)) * d.cbs, cp.flogits, d.cbs);
    if (threadIdx.x == 0 && c < d.ncb - 1) cp.fcode[c] = checked_id(cp, cp.fin_prefix[f * (d.ncb - 1) + c], d.cbs);
    return;
  }
  if (cp.dbg_fast) copy_vec(cp.dbg_fast + (static_cast<size_t>(f) * (d.ncb - 1) + (c - 1)) * d.cbs, cp.flogits, d.cbs);
  const float* E = cp.expo + static_cast<size_t>(f) * kDraws * kTopK + (1 + c) * kTopK;
  int dc = draw(cp.d, *reinterpret_cast<SampScratch*>(S.xs), cp.flogits, d.cbs, false, false, cp.temperature, cp.top_p, E);
  if (threadIdx.x == 0) {
    if (cp.dbg_draws) cp.dbg_draws[f * kDraws + 1 + c] = dc;
    if (cp.forced) dc = checked_id(cp, cp.forced[f * kDraws + 1 + c], d.cbs);
    if (dc < 0) dc = 0;  // nothing drawable: the remaining codes are 0 (ch.06 §5.2)
    cp.fcode[c] = dc;
    cp.st->vals[1 + c] = dc;
    cp.stage[static_cast<size_t>(f) * d.ncb + c] = dc;
    if (c == d.ncb - 1) cp.st->n_out = f + 1;
  }
}

// Fast-AR-alone mode: the frame's hidden and first prefix code (CTA 0)
__device__ void fast_in(const CallParams& cp, int f) {
  const Dims& d = cp.d;
  for (int i = threadIdx.x; i < d.D; i += kConsumers) cp.hidden[i] = cp.fin_hidden[static_cast<size_t>(f) * d.D + i];
  if (threadIdx.x == 0) cp.fcode[0] = checked_id(cp, cp.fin_prefix[f * (d.ncb - 1)], d.cbs);
}

// =========================================================================
// consumers
// =========================================================================

template <class C>
__device__ void consumers(const CallParams& cp, Smem& S) {
  Pipe pipe{0, 0, 0, 0u};
  unsigned target = cp.gbar_base;  // the host starts the counter there
  const bool cta0 = blockIdx.x == 0;
  const int tid = threadIdx.x;
  constexpr int NQ = static_cast<int>(sizeof(Phase) / 16);
  if (!cp.fast_only && ldcgi(&cp.st->done) != 0) {
    if (cta0 && tid == 0) cp.st->n_out = 0;
    return;
  }
  if (cta0 && tid == 0) cp.st->n_out = 0;
  // phase descriptors live in shared memory; the next one is fetched while the current one runs
  if (tid < NQ) reinterpret_cast<uint4*>(&S.ph[0])[tid] = __ldg(reinterpret_cast<const uint4*>(cp.prog) + tid);
  // the stream position advances by one per frame (the last phase of a frame bumps it), so the
  // slot of frame f is the position at the launch + f: read once here, not in every layer
  const int pos_launch = cp.fast_only ? 0 : ldcgi(&cp.st->pos);
  if (tid == 0) {
    // the Fast-AR attention item of this CTA, fixed for the launch (no division per phase)
    S.fa_rep = cp.d.Hqf / cp.d.Hkvf;
    S.fa_j = static_cast<int>(blockIdx.x) / cp.d.Hqf;
    S.fa_h = static_cast<int>(blockIdx.x) % cp.d.Hqf;
    S.fa_g = S.fa_h / S.fa_rep;
  }
  named_bar(1, kConsumers);
  int k = 0;
  for (int f = 0; f < cp.n_frames; ++f) {
    if (tid == 0) {
      // the Slow-AR attention plan depends on the frame's slot only: its integer divisions are
      // taken once per frame, not in every layer
      S.pos_frame = pos_launch + f;
      if (!cp.fast_only && cp.d.L > 0) {
        int ns, chunk;
        attn_split(pos_launch + f + 1, static_cast<int>(gridDim.x), cp.d.Hkv, ns, chunk);
        S.attn_ns = ns;
        S.attn_chunk = chunk;
        S.attn_g = static_cast<int>(blockIdx.x) / ns;
        S.attn_s = static_cast<int>(blockIdx.x) % ns;
        S.attn_rep = cp.d.Hq / cp.d.Hkv;
        S.attn_pml = attn_part_ml(cp, static_cast<int>(gridDim.x));
      }
    }
    for (int p = 0; p < cp.n_phases; ++p, ++k) {
      const Phase& ph = S.ph[k & 1];
      int np = p + 1;
      if (np == cp.n_phases) np = 0;
      const bool has_next = (p + 1 < cp.n_phases) || (f + 1 < cp.n_frames);
      // the next descriptor travels into the other slot while this phase runs (an async copy, so
      // that no register holds it and its load is not deferred to the end of the phase)
      if (tid < NQ && has_next)
        cp_async16(reinterpret_cast<uint4*>(&S.ph[(k + 1) & 1]) + tid, reinterpret_cast<const uint4*>(cp.prog + np) + tid);
      pipe.tag = cp.tag0 + static_cast<uint32_t>(k);
      if (tid == 0) S.phase_k = k;
      switch (ph.op) {
        case OP_GEMV:
          if (ph.merge_main && cta0) sample_main(cp, S, f);
          else pipe = gemv<C>(cp, ph, S, pipe);
          break;
        case OP_ATTN_SLOW:
          attn_slow<C>(cp, ph, S, pipe.tag);
          break;
        case OP_ATTN_FAST:
          attn_fast<C>(cp, ph, S, pipe.tag);
          break;
        case OP_SAMPLE_FAST:
          if (cta0) sample_fast(cp, S, f, ph.cb);
          break;
        case OP_SAMPLE_MAIN:
          if (cta0) sample_main(cp, S, f);
          break;
        case OP_FAST_IN:
          if (cta0) fast_in(cp, f);
          break;
        default:
          break;
      }
      if (ph.bump_pos && cta0 && tid == 0) {
        cp.st->pos = cp.st->pos + 1;  // the Slow-AR step's last phase: its slot is now filled
      }
      if (tid < NQ) cp_async_wait_all();
      if (ph.no_sync) {
        // the next phase polls this phase's tagged outputs: only this CTA's threads meet here
        named_bar(1, kConsumers);
        if (*reinterpret_cast<volatile int*>(&S.fail) != 0) return;
      } else if (!grid_sync(cp, S, target)) {
        return;
      }
      if (cp.trace != nullptr && cta0 && tid == 0) {
        const int kk = f * cp.n_phases + p;
        if (kk < cp.trace_cap) cp.trace[kk] = globaltimer_ns();
      }
      if ((ph.op == OP_SAMPLE_MAIN || ph.merge_main) && ldcgi(&cp.st->done) != 0) return;
    }
  }
}

template <class C>
__global__ void __launch_bounds__(kThreads, 1) frame_kernel(const __grid_constant__ CallParams params) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  Smem& S = *reinterpret_cast<Smem*>(smem_raw);
  static_assert(sizeof(CallParams) % 16 == 0, "parameter copy");
  for (int i = threadIdx.x; i < static_cast<int>(sizeof(CallParams) / 16); i += kThreads)
    reinterpret_cast<uint4*>(&S.cp)[i] = reinterpret_cast<const uint4*>(&params)[i];
  const CallParams& cp = S.cp;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], kConsumerWarps);
    }
    mbar_init(&S.xsbar, 1);
    S.abort_flag = 0;
    S.fail = 0;
    S.sync_ok = 1;
    S.flag = 0;
    S.phase_k = -1;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x >= kConsumers) {
    producer<C>(cp, S);
  } else {
    consumers<C>(cp, S);
    named_bar(1, kConsumers);
    if (threadIdx.x == 0) {
      __threadfence_block();
      *reinterpret_cast<volatile int*>(&S.abort_flag) = 1;
    }
  }
}

}  // namespace
}  // namespace s2
