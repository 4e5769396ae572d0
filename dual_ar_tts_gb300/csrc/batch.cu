// Batched frame decode: one decode call advances B independent streams together, and every weight
// matrix is read from HBM once per step for the whole batch (the frame loop of s2.cpp analysis
// ch.06 §5.1 run for B streams at once; the projections of ch.02 §3.2 as skinny GEMMs).
//
// One frame is a fixed sequence of kernels, captured once per call as a CUDA graph and replayed
// for every frame (kernels read the frame index from device memory):
//
//   main draws (one CTA per stream) -> fast_project_in -> Fast-AR calls 1..9 (4 layers each, then
//   fast_output and the draw) -> Slow-AR step (36 layers, final norm, admissible tied logits)
//
// Projections run on the 5th-generation tensor cores (k_bgemv): y[c] = W·a_c for the NC columns
// of the batch.  Tiles of 128 weight rows × 64 K come in by TMA (128-byte swizzle); the
// activations are bf16 hi/lo "planes" (row 2c = hi, row 2c+1 = lo, hi + lo = the fp32 value to
// ~2^-17), the MMA's N dimension; one thread issues tcgen05.mma into a TMEM accumulator and four
// warps read it back.  K is split across CTAs so that every SM streams weights; the partial sums
// are reduced in a fixed order by the consumer kernel (deterministic results).  The consumer
// kernels fuse what follows a projection: residual add + RMSNorm + planes for the next
// projection, SwiGLU, q/k norm + RoPE + KV store + attention, the draws.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <map>
#include <string>
#include <tuple>
#include <vector>

#include "ptx.cuh"
#include "s2_internal.h"
#include "sampler.cuh"
#include "tc05.cuh"

namespace s2 {
namespace {

constexpr int kTileM = 128;                 // weight rows per MMA tile (the MMA's M)
constexpr int kAtom = 64;                   // K elements per pipeline stage (one 128-byte row)
constexpr int kABytes = kTileM * kAtom * 2;  // one weight tile
constexpr int kGemvThreads = 192;           // 4 epilogue warps, 1 TMA warp, 1 MMA warp
constexpr int kMaxGemvStages = 8;
constexpr int kGemvSmemBudget = 100 * 1024;  // two CTAs per SM
constexpr int kGemvCtasPerSm = 2;
// dynamic shared memory of a projection CTA is at least this much, so that no more than two of
// them (each holding up to 256 TMEM columns of the SM's 512) are ever resident on one SM
constexpr int kGemvSmemFloor = 80 * 1024;
constexpr int kSamplerSplits = 4;             // split-K of projections summed by one CTA per stream
constexpr int kPrefillCols = 128;             // prompt positions per projection launch (N = 256)
constexpr int kPrepThreads = 1024;                // column preparation: one CTA per column
constexpr int kPrepPer = 3;                       // row elements per thread
constexpr int kPrepMaxK = kPrepPer * kPrepThreads;  // longest row a column-preparation CTA holds
constexpr int kAttnChunk = 1024;            // target slots per Slow-AR attention item
constexpr int kAttnStages = 3;              // K/V slot groups in flight per warp
constexpr int kMaxSplitsAttn = 32;          // items per (stream, KV head) at most

enum ColMode : int { CM_RESID = 0, CM_STORE, CM_FEROW, CM_EMBED, CM_HIDDEN };

// per-stream settings of a call (device copy)
struct BStream {
  int sid, min_tokens, ras_window, pad;
  float T, top_p, ras_T, ras_top_p;
  const float* expo;       // [n_frames][11][30]
  const int32_t* forced;   // [n_frames][11] or null
  float* dbg_main;         // [n_frames][A] or null
  float* dbg_fast;         // [n_frames][NCB-1][CBS] or null
  float* dbg_hidden;       // [n_frames][D] or null
  int32_t* dbg_draws;      // [n_frames][11] or null
};

// everything a batched kernel may touch (passed by value)
struct BEnv {
  Dims d;
  int nb;
  int max_streams, kv_slots, lstride;
  StreamState* st;
  const BStream* bs;
  int* bctl;               // [0] frame index within the call
  float* hidden;           // [max_streams][D]
  float* logits;           // [max_streams][lstride]
  int32_t* stage;          // [max_streams][kMaxFramesPerCall][NCB]
  Control* ctl;
  unsigned char* kc;
  unsigned char* vc;
  const float2* rope;
  const float2* rope_f;
  const void* E;
  const void* CE;
  const void* FE;
  uint16_t* pX;            // planes [rows][ldX]
  uint16_t* pO;
  uint16_t* pH;
  int ldX, ldO, ldH;
  float* part;             // split-K partials
  float* bx;               // [max_streams][D]       Slow-AR residual
  float* bfx;              // [max_streams][2][Df]   Fast-AR residual rows of the call's new positions
  float* bfk;              // [max_streams][Lf][Wf][Hkvf][hdf]
  float* bfv;
  float* apart;            // attention split partials
  float* bflog;            // [max_streams][CBS]
  int32_t* bfcode;         // [max_streams][16]
};

__device__ __forceinline__ int frame_index(const BEnv& e) { return ldcgi(e.bctl); }
__device__ __forceinline__ bool stream_done(const BEnv& e, int sid) { return ldcgi(&e.st[sid].done) != 0; }

__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, Control* ctl) {
  const long long lim = ctl->spin_limit;
  const long long t0 = clock_us();
  for (unsigned i = 1;; ++i) {
    if (mbar_test(bar, parity)) return true;
    if ((i & 255u) == 0 && clock_us() - t0 > lim) break;
  }
  if (atomicCAS(&ctl->error, 0, S2_ETIMEOUT) == 0) ctl->error_where = 10;
  return false;
}

__device__ __forceinline__ void store_hilo(uint16_t* planes, int ld, int col, int k, float v) {
  const __nv_bfloat16 hi = __float2bfloat16_rn(v);
  const __nv_bfloat16 lo = __float2bfloat16_rn(v - __bfloat162float(hi));
  planes[static_cast<size_t>(2 * col) * ld + k] = __bfloat16_as_ushort(hi);
  planes[static_cast<size_t>(2 * col + 1) * ld + k] = __bfloat16_as_ushort(lo);
}

// deterministic block sum (fixed order) over the NT threads of the block; red holds NT / 32 floats
template <int NT>
__device__ __forceinline__ float block_sum(float v, float* red) {
  v = warp_sum(v);
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[w] = v;
  __syncthreads();
  float t = 0.f;
#pragma unroll
  for (int i = 0; i < NT / 32; ++i) t += red[i];
  return t;
}

// =========================================================================================
// projection: part[((z*splits + split)*NC + c)*M + m] = Σ_{k in split} W_z[row0 + m][k]·a_c[k]
// =========================================================================================

struct GemvBars {
  uint64_t full[kMaxGemvStages], empty[kMaxGemvStages], acc;
  uint32_t taddr;
};

__global__ void __launch_bounds__(kGemvThreads, kGemvCtasPerSm)
    k_bgemv(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmA2,
            const __grid_constant__ CUtensorMap tmB, int M, int row0, int N, int NC, int atoms_total, int atoms_per,
            int nstages, float* part, Control* ctl) {
  extern __shared__ __align__(1024) unsigned char smraw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
  const int sbytes = kABytes + N * 128;
  GemvBars& S = *reinterpret_cast<GemvBars*>(sm + nstages * sbytes);
  const int tile = blockIdx.x, split = blockIdx.y, z = blockIdx.z, splits = gridDim.y;
  const int a0 = split * atoms_per, a1 = min(a0 + atoms_per, atoms_total);
  const int na = a1 - a0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const CUtensorMap* tA = z == 0 ? &tmA : &tmA2;
  pdl_trigger();
  if (threadIdx.x == 0) {
    for (int s = 0; s < nstages; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], 1);
    }
    mbar_init(&S.acc, 1);
    fence_barrier_init();
  }
  const uint32_t ncols = N <= 32 ? 32u : (N <= 64 ? 64u : (N <= 128 ? 128u : 256u));
  if (warp == 0) {
    tmem_alloc(&S.taddr, ncols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tacc = S.taddr;
  if (warp == 4) {
    if (lane == 0) {
      prefetch_tmap(tA);
      prefetch_tmap(&tmB);
      const uint64_t pol = policy_evict_first();
      // the weights do not depend on earlier kernels: the first stages' weight tiles are requested
      // before waiting for the grid that produces the activations
      const int pre = min(nstages, na);
      for (int i = 0; i < pre; ++i) {
        mbar_arrive_expect_tx(&S.full[i], sbytes);
        tma_load_2d(sm + i * sbytes, tA, (a0 + i) * kAtom, row0 + tile * kTileM, &S.full[i], pol);
      }
      pdl_wait();
      for (int i = 0; i < pre; ++i)
        tma_load_2d(sm + i * sbytes + kABytes, &tmB, (a0 + i) * kAtom, 0, &S.full[i], pol);
      for (int i = pre; i < na; ++i) {
        const int s = i % nstages;
        if (!wait_bar(&S.empty[s], ((i / nstages) & 1) ^ 1, ctl)) break;
        unsigned char* A = sm + s * sbytes;
        mbar_arrive_expect_tx(&S.full[s], sbytes);
        tma_load_2d(A, tA, (a0 + i) * kAtom, row0 + tile * kTileM, &S.full[s], pol);
        tma_load_2d(A + kABytes, &tmB, (a0 + i) * kAtom, 0, &S.full[s], pol);
      }
    }
  } else if (warp == 5) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(kTileM, N);
      int i = 0;
      for (; i < na; ++i) {
        const int s = i % nstages;
        if (!wait_bar(&S.full[s], (i / nstages) & 1, ctl)) break;
        tc_fence_after();
        const uint32_t A = smem_u32(sm + s * sbytes);
        const uint32_t B = A + kABytes;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          tc_mma(tacc, desc_sw128(A + kk * 32), desc_sw128(B + kk * 32), idesc, (i > 0 || kk > 0) ? 1u : 0u);
        tc_commit(&S.empty[s]);
      }
      tc_commit(&S.acc);
    }
  } else {
    const bool ok = __all_sync(0xffffffffu, wait_bar(&S.acc, 0, ctl));
    pdl_wait();  // the partials buffer may still be read by the previous grid until it completes
    if (ok) {
      tc_fence_after();
      const int row = tile * kTileM + warp * 32 + lane;
      float* out = part + (static_cast<size_t>(z) * splits + split) * NC * M;
      for (int c0 = 0; c0 < N; c0 += 16) {
        float v[16];
        tmem_ld16(tacc + (static_cast<uint32_t>(warp * 32) << 16) + c0, v);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int c = c0 / 2 + j;
          if (c < NC && row < M) out[static_cast<size_t>(c) * M + row] = v[2 * j] + v[2 * j + 1];
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tacc, ncols);
}

// =========================================================================================
// fp8 projection: the same partials from e4m3 weights Q with one fp32 scale per row,
// part[...] = scale[row0 + m]·Σ_{k in split} Q[row0 + m][k]·a_c[k].  K advances 128 per step (one
// 128-byte fp8 row per weight row, 128-byte swizzle).  Two rings: fp8 weight tiles, and the planes
// of the same 128 K (two 64-K boxes).  Eight warps, idle until the accumulator is ready, expand
// each fp8 tile to bf16 in registers (a thread owns one tile row = one TMEM lane, half of its 128
// codes) and store it into one of the tensor-memory A buffers, from which the MMA reads A (B, the
// planes, stays in shared memory).  A weight slot is refilled as soon as its tile has been read;
// a planes slot and an A buffer once the MMAs that read them have completed.
// =========================================================================================

constexpr int kAtom8 = 128;                // K elements per fp8 step
constexpr int kA8Bytes = kTileM * kAtom8;  // one fp8 weight tile (16 KB)
constexpr int kGemv8Threads = 320;         // 8 expanding / epilogue warps, a TMA warp, an MMA warp
constexpr int kMaxTBufs = 4;               // tensor-memory A buffers at most

struct Gemv8Bars {
  uint64_t wfull[kMaxGemvStages], wempty[kMaxGemvStages];  // fp8 weight tiles
  uint64_t bfull[kMaxGemvStages], bempty[kMaxGemvStages];  // planes
  uint64_t tfull[kMaxTBufs], tempty[kMaxTBufs];            // tensor-memory A buffers
  uint64_t acc;
  uint32_t taddr;
};

// tensor memory: accumulator columns [0, acc), then A buffers of 64 columns up to the allocation
__host__ __device__ constexpr int gemv8_acc_cols(int N) { return N <= 64 ? 64 : (N <= 128 ? 128 : 256); }
__host__ __device__ constexpr int gemv8_tmem_cols(int N) { return N <= 128 ? 256 : 512; }
__host__ __device__ constexpr int gemv8_tbufs(int N) {
  const int n = (gemv8_tmem_cols(N) - gemv8_acc_cols(N)) / 64;
  return n < kMaxTBufs ? n : kMaxTBufs;
}

__global__ void __launch_bounds__(kGemv8Threads, kGemvCtasPerSm)
    k_bgemv8(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmA2,
             const __grid_constant__ CUtensorMap tmB, const float* scA, const float* scA2, int M, int row0, int N,
             int NC, int atoms_total, int atoms_per, int nw, int nb, float* part, Control* ctl) {
  extern __shared__ __align__(1024) unsigned char smraw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
  const int bbytes = N * 128;  // planes of 64 K
  unsigned char* smW = sm;
  unsigned char* smB = sm + nw * kA8Bytes;
  Gemv8Bars& S = *reinterpret_cast<Gemv8Bars*>(smB + nb * 2 * bbytes);
  const int tile = blockIdx.x, split = blockIdx.y, z = blockIdx.z, splits = gridDim.y;
  const int a0 = split * atoms_per, a1 = min(a0 + atoms_per, atoms_total);
  const int na = a1 - a0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const CUtensorMap* tA = z == 0 ? &tmA : &tmA2;
  const float* sc = z == 0 ? scA : scA2;
  const int acc_cols = gemv8_acc_cols(N), ncols = gemv8_tmem_cols(N), nt = gemv8_tbufs(N);
  pdl_trigger();
  if (threadIdx.x == 0) {
    for (int s = 0; s < nw; ++s) {
      mbar_init(&S.wfull[s], 1);
      mbar_init(&S.wempty[s], 8);  // the eight expanding warps
    }
    for (int s = 0; s < nb; ++s) {
      mbar_init(&S.bfull[s], 1);
      mbar_init(&S.bempty[s], 1);  // the MMA's commit
    }
    for (int b = 0; b < nt; ++b) {
      mbar_init(&S.tfull[b], 8);
      mbar_init(&S.tempty[b], 1);
    }
    mbar_init(&S.acc, 1);
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(&S.taddr, static_cast<uint32_t>(ncols));
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tacc = S.taddr;
  if (warp == 8) {
    if (lane == 0) {
      // weight tiles: independent of earlier kernels, requested without waiting for them
      prefetch_tmap(tA);
      const uint64_t pol = policy_evict_first();
      for (int i = 0; i < na; ++i) {
        const int s = i % nw;
        if (i >= nw && !wait_bar(&S.wempty[s], ((i / nw) & 1) ^ 1, ctl)) break;
        mbar_arrive_expect_tx(&S.wfull[s], kA8Bytes);
        tma_load_2d(smW + s * kA8Bytes, tA, (a0 + i) * kAtom8, row0 + tile * kTileM, &S.wfull[s], pol);
      }
    } else if (lane == 1) {
      // planes: produced by the previous kernel; shared by every row tile of this split
      prefetch_tmap(&tmB);
      const uint64_t pol = policy_evict_last();
      pdl_wait();
      for (int i = 0; i < na; ++i) {
        const int s = i % nb;
        if (i >= nb && !wait_bar(&S.bempty[s], ((i / nb) & 1) ^ 1, ctl)) break;
        unsigned char* Bs = smB + s * 2 * bbytes;
        mbar_arrive_expect_tx(&S.bfull[s], 2 * bbytes);
        tma_load_2d(Bs, &tmB, (a0 + i) * kAtom8, 0, &S.bfull[s], pol);
        tma_load_2d(Bs + bbytes, &tmB, (a0 + i) * kAtom8 + kAtom, 0, &S.bfull[s], pol);
      }
    }
  } else if (warp == 9) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(kTileM, N);
      for (int i = 0; i < na; ++i) {
        const int s = i % nb, b = i % nt;
        if (!wait_bar(&S.tfull[b], (i / nt) & 1, ctl)) break;
        if (!wait_bar(&S.bfull[s], (i / nb) & 1, ctl)) break;
        tc_fence_after();
        const uint32_t B = smem_u32(smB + s * 2 * bbytes);
        const uint32_t abuf = tacc + static_cast<uint32_t>(acc_cols + b * 64);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          tc_mma_tmem_a(tacc, abuf + kk * 8, desc_sw128(B + (kk >> 2) * bbytes + (kk & 3) * 32), idesc,
                        (i > 0 || kk > 0) ? 1u : 0u);
        tc_commit(&S.bempty[s]);
        tc_commit(&S.tempty[b]);
      }
      tc_commit(&S.acc);
    }
  } else {
    // warps 0..7: warp w expands half h = w / 4 (codes 64h .. 64h + 63) of tile rows 32q .. 32q + 31,
    // q = w % 4 (the TMEM lane quarter this warp may access)
    const int q = warp & 3, h = warp >> 2;
    const int r = q * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    for (int i = 0; i < na; ++i) {
      const int s = i % nw, b = i % nt;
      if (!__all_sync(0xffffffffu, wait_bar(&S.wfull[s], (i / nw) & 1, ctl))) break;
      if (!__all_sync(0xffffffffu, wait_bar(&S.tempty[b], ((i / nt) & 1) ^ 1, ctl))) break;
      tc_fence_after();
      const unsigned char* rowp = smW + s * kA8Bytes + r * 128;
      uint32_t o[32];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int chunk = h * 4 + c;  // K elements 16·chunk .. 16·chunk + 15
        const uint4 w = *reinterpret_cast<const uint4*>(rowp + ((chunk ^ (r & 7)) << 4));
        e4m3x4_to_bf16x4(w.x, o[c * 8 + 0], o[c * 8 + 1]);
        e4m3x4_to_bf16x4(w.y, o[c * 8 + 2], o[c * 8 + 3]);
        e4m3x4_to_bf16x4(w.z, o[c * 8 + 4], o[c * 8 + 5]);
        e4m3x4_to_bf16x4(w.w, o[c * 8 + 6], o[c * 8 + 7]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.wempty[s]);  // the weight slot's codes are in registers
      tmem_st32(tacc + lane_off + static_cast<uint32_t>(acc_cols + b * 64 + h * 32), o);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.tfull[b]);
    }
    const bool ok = __all_sync(0xffffffffu, wait_bar(&S.acc, 0, ctl));
    pdl_wait();  // the partials buffer may still be read by the previous grid until it completes
    if (ok) {
      tc_fence_after();
      const int row = tile * kTileM + r;
      const float scale = row < M ? __ldg(sc + row0 + row) : 0.f;
      float* out = part + (static_cast<size_t>(z) * splits + split) * NC * M;
      for (int c0 = h * 16; c0 < N; c0 += 32) {
        float v[16];
        tmem_ld16(tacc + lane_off + c0, v);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int c = c0 / 2 + j;
          if (c < NC && row < M) out[static_cast<size_t>(c) * M + row] = (v[2 * j] + v[2 * j + 1]) * scale;
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tacc, static_cast<uint32_t>(ncols));
}

// =========================================================================================
// e4m3 quantisation of bf16 rows: scale = max|w| / 448 (fp32 division), code = w / scale rounded
// to the nearest e4m3 value, ties to even, saturating at ±448; an all-zero row gets scale 0 and
// zero codes.  One CTA per row (grid-stride).
constexpr int kQuantThreads = 256;

__global__ void __launch_bounds__(kQuantThreads) k_quant_e4m3(const uint16_t* w, long long rows, int K, uint8_t* q,
                                                              float* scales) {
  __shared__ float red[kQuantThreads / 32];
  for (long long r = blockIdx.x; r < rows; r += gridDim.x) {
    const uint16_t* wr = w + r * K;
    float m = 0.f;
    for (int k = threadIdx.x; k < K; k += kQuantThreads) m = fmaxf(m, fabsf(bf16_to_f(wr[k])));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < kQuantThreads / 32; ++i) amax = fmaxf(amax, red[i]);
    __syncthreads();
    const float scale = __fdiv_rn(amax, 448.f);
    if (threadIdx.x == 0) scales[r] = scale;
    uint8_t* qr = q + r * K;
    for (int k = threadIdx.x; k < K; k += kQuantThreads) {
      uint8_t code = 0;
      if (scale > 0.f) {
        const float v = __fdiv_rn(bf16_to_f(wr[k]), scale);
        uint16_t pair;  // v converted into both bytes
        asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(pair) : "f"(v), "f"(v));
        code = static_cast<uint8_t>(pair & 0xFFu);
      }
      qr[k] = code;
    }
  }
}

// Check of the e4m3 -> bf16 expansion used by k_bgemv8 against the hardware e4m3 -> f16
// conversion, over every finite code: bad[0] = number of codes that differ.
__global__ void k_e4m3_selfcheck(int* bad) {
  const uint32_t c = threadIdx.x;  // 256 threads, one code each
  if ((c & 0x7Fu) == 0x7Fu) return;  // NaN codes are never produced
  uint32_t lo, hi;
  e4m3x4_to_bf16x4(c | (c << 8) | (c << 16) | (c << 24), lo, hi);
  uint32_t h2;
  const uint16_t in = static_cast<uint16_t>(c | (c << 8));
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(in));
  const float ref = __half2float(__ushort_as_half(static_cast<uint16_t>(h2 & 0xFFFFu)));
  const float got[4] = {bf16lo(lo), bf16hi(lo), bf16lo(hi), bf16hi(hi)};
  bool ok = true;
  for (int i = 0; i < 4; ++i)
    ok = ok && __float_as_uint(got[i]) == __float_as_uint(ref);
  if (!ok) atomicAdd(bad, 1);
}

// =========================================================================================
// column preparation: the fp32 input row of each column (residual add of split partials, a
// fast_embeddings row, the Slow-AR input embedding, or the hidden state), stored, RMS-normalised
// with a norm weight, and written as hi/lo planes for the next projection
// =========================================================================================

struct ColPrep {
  int npos;               // columns per stream
  int mode[2];            // ColMode of position j
  int K;                  // row length
  const float* part;      // partials [splits][part_nc][K] (CM_RESID, CM_STORE)
  int splits;
  int part_nc;            // columns of the partials
  int part_by_stream;     // partial column = stream b (else = this column c)
  float* x;               // residual rows: stream b, position j at x + b*xb + j*K
  int xb;
  const void* normw;      // RMSNorm weight (bf16 or fp32 per d.esz); null: no norm
  int last_only;          // planes only for position npos-1, at column b
  int code_idx;           // CM_FEROW: which code of the frame (bfcode[b][code_idx])
  float* hid_out;         // optional: the normalised row (by stream id, stride D)
};

__global__ void __launch_bounds__(kPrepThreads) k_colprep(const BEnv e, const ColPrep p) {
  pdl_wait();
  pdl_trigger();
  __shared__ float red[kPrepThreads / 32];
  constexpr int kMaxPer = kPrepPer;  // K <= kPrepMaxK (checked on the host)
  const Dims& d = e.d;
  const int c = blockIdx.x, b = c / p.npos, j = c % p.npos;
  const int sid = e.bs[b].sid;
  if (stream_done(e, sid)) return;
  const int K = p.K, tid = threadIdx.x;
  const int mode = p.mode[j];
  const int pcol = p.part_by_stream ? b : c;
  float v[kMaxPer];
#pragma unroll
  for (int i = 0; i < kMaxPer; ++i) v[i] = 0.f;
  float ss = 0.f;
  int code = 0, tok = 0;
  float msem = 0.f;
  if (mode == CM_FEROW) code = ldcgi(&e.bfcode[b * 16 + p.code_idx]);
  if (mode == CM_EMBED) {
    tok = ldcgi(&e.st[sid].vals[0]);
    msem = (tok >= d.sem_lo && tok <= d.sem_hi) ? 1.f : 0.f;
  }
  float* xr = p.x ? p.x + static_cast<size_t>(b) * p.xb + static_cast<size_t>(j) * K : nullptr;
  // gather every input first (no stores in between, so the loads overlap), then store
  if (mode == CM_RESID || mode == CM_STORE) {
#pragma unroll
    for (int i = 0; i < kMaxPer; ++i) {
      const int k = tid + i * kPrepThreads;
      v[i] = (mode == CM_RESID && k < K) ? __ldcg(xr + k) : 0.f;
    }
    // eight splits per round: their loads are issued together (the sums keep split order)
    constexpr int SR = 8;
    const size_t sstride = static_cast<size_t>(p.part_nc) * K;
    const float* pc = p.part + static_cast<size_t>(pcol) * K;
    for (int s = 0; s < p.splits; s += SR) {
      float t[SR][kMaxPer];
#pragma unroll
      for (int j = 0; j < SR; ++j)
#pragma unroll
        for (int i = 0; i < kMaxPer; ++i) {
          const int k = tid + i * kPrepThreads;
          t[j][i] = (s + j < p.splits && k < K) ? __ldcg(pc + (s + j) * sstride + k) : 0.f;
        }
#pragma unroll
      for (int j = 0; j < SR; ++j)
#pragma unroll
        for (int i = 0; i < kMaxPer; ++i) v[i] += t[j][i];
    }
  }
#pragma unroll
  for (int i = 0; i < kMaxPer; ++i) {
    const int k = tid + i * kPrepThreads;
    float a = v[i];
    if (k < K) {
      if (mode == CM_RESID || mode == CM_STORE) {
      } else if (mode == CM_FEROW) {
        a = wload(e.FE, static_cast<size_t>(code) * K + k, d.esz);
      } else if (mode == CM_EMBED) {
        // x = sem_scale·E[r0] + m·Σ_cb CE[cb·CBS + code_cb]   (ch.02 §3.2)
        float acc = 0.f;
        for (int cb = 0; cb < d.ncb; ++cb) {
          const size_t row = static_cast<size_t>(cb) * d.cbs + ldcgi(&e.st[sid].vals[1 + cb]);
          acc = __fadd_rn(acc, wload(e.CE, row * K + k, d.esz));
        }
        a = __fadd_rn(__fmul_rn(d.sem_scale, wload(e.E, static_cast<size_t>(tok) * K + k, d.esz)), __fmul_rn(msem, acc));
      } else {  // CM_HIDDEN
        a = __ldcg(e.hidden + static_cast<size_t>(sid) * d.D + k);
      }
    }
    v[i] = a;
  }
#pragma unroll
  for (int i = 0; i < kMaxPer; ++i) {
    const int k = tid + i * kPrepThreads;
    if (k < K) {
      if (xr) xr[k] = v[i];
      ss += v[i] * v[i];
    }
  }
  float r = 1.f;
  if (p.normw) r = 1.0f / sqrtf(block_sum<kPrepThreads>(ss, red) / static_cast<float>(K) + d.eps);
  const bool planes = !p.last_only || j == p.npos - 1;
  const int pc = p.last_only ? b : c;
#pragma unroll
  for (int i = 0; i < kMaxPer; ++i) {
    const int k = tid + i * kPrepThreads;
    if (k < K) {
      const float n = p.normw ? (v[i] * r) * wload(p.normw, k, d.esz) : v[i];
      if (planes) store_hilo(e.pX, e.ldX, pc, k, n);
      if (p.hid_out) p.hid_out[static_cast<size_t>(sid) * d.D + k] = n;
    }
  }
}

// SwiGLU of the two projections (split partials of W1, then of W3): planes of silu(g)·u
__global__ void __launch_bounds__(256) k_swiglu(const BEnv e, const float* __restrict__ part, int M, int NC,
                                                int splits) {
  pdl_wait();
  pdl_trigger();
  const int c = blockIdx.y;
  const int sid = e.bs[c / (NC / e.nb)].sid;
  if (stream_done(e, sid)) return;
  for (int m = blockIdx.x * blockDim.x + threadIdx.x; m < M; m += gridDim.x * blockDim.x) {
    float a = 0.f, u = 0.f;
    for (int s = 0; s < splits; ++s) {
      a += __ldcg(part + (static_cast<size_t>(s) * NC + c) * M + m);
      u += __ldcg(part + (static_cast<size_t>(splits + s) * NC + c) * M + m);
    }
    store_hilo(e.pH, e.ldH, c, m, (a / (1.0f + expf(-a))) * u);
  }
}

// =========================================================================================
// attention
// =========================================================================================

template <typename KT>
__device__ __forceinline__ float kvf(KT x);
template <>
__device__ __forceinline__ float kvf<__half>(__half x) { return __half2float(x); }
template <typename KT>
__device__ __forceinline__ KT tokv(float x);
template <>
__device__ __forceinline__ __half tokv<__half>(float x) { return __float2half_rn(x); }

// per-head RMSNorm (weight [hd]) then RoPE on adjacent pairs, in place on v[0..HD) by 128 threads
// of one head group (helpers run by the whole CTA with head h = thread / (HD/2) pairs)
template <int HD>
__device__ void norm_rope_heads(float* v, int nheads, const void* nw, bool norm, int esz, float eps,
                                const float2* rope_row, float* red) {
  // v: [nheads][HD] in shared memory; thread t handles pair (h, i) for t < nheads*HD/2
  const int tid = threadIdx.x;
  constexpr int P = HD / 2;
  __syncthreads();
  if (norm) {
    // sum of squares per head: one warp per head
    const int w = tid >> 5, lane = tid & 31;
    for (int h = w; h < nheads; h += blockDim.x >> 5) {
      float s = 0.f;
      for (int i = lane; i < HD; i += 32) s += v[h * HD + i] * v[h * HD + i];
      s = warp_sum(s);
      if (lane == 0) red[h] = 1.0f / sqrtf(s / static_cast<float>(HD) + eps);
    }
    __syncthreads();
  }
  for (int t = tid; t < nheads * P; t += blockDim.x) {
    const int h = t / P, i = t % P;
    float a = v[h * HD + 2 * i], bb = v[h * HD + 2 * i + 1];
    if (norm) {
      a = (a * red[h]) * wload(nw, 2 * i, esz);
      bb = (bb * red[h]) * wload(nw, 2 * i + 1, esz);
    }
    const float2 cs = rope_row[i];
    v[h * HD + 2 * i] = a * cs.x - bb * cs.y;
    v[h * HD + 2 * i + 1] = a * cs.y + bb * cs.x;
  }
  __syncthreads();
}

// tensor-core fragments (mma.sync m16n8k16, fp16 inputs, fp32 accumulation)
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a2, uint32_t b0, uint32_t b1) {
  // rows 8..15 of A are zero (a1 = a3 = 0)
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_f16x(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}
// x split as fp16 hi (part 0) or the fp16 remainder x - hi (part 1)
__device__ __forceinline__ float h_part(float x, int part) {
  const float hi = __half2float(__float2half_rn(x));
  return part == 0 ? hi : x - hi;
}

// Slow-AR: item (stream b, KV head g, split s) over its range of slots; the item whose range
// holds the new slot normalises, rotates and stores the new K/V first.  Each of the 4 warps owns
// every fourth group of 16 slots of the range and runs its own cp.async pipeline, online softmax
// and P·V, so the slot loop needs no block-wide barrier; the warps' results are combined at the
// end.  Scores and P·V run on the tensor cores (mma.sync, fp16 inputs, fp32 accumulation):
//   S = [q_hi; q_lo] · K^T   rows 0-3 / 4-7 of A = fp16 hi / remainder of the 4 scaled query
//                            heads (q = hi + lo to ~2^-22), B = the fp16 K rows (ldmatrix)
//   O += [p_hi; p_lo] · V    A = the probabilities (hi / remainder) taken from the score
//                            accumulators' registers, B = the fp16 V rows (ldmatrix.trans)
// and the hi and lo rows are added at the end, so the result carries fp32 precision.
template <int HD, typename KT>
__global__ void __launch_bounds__(128, 2) k_attn_slow(const BEnv e, int layer, const void* qn, const void* kn,
                                                      const float* __restrict__ part, int splits, int ns, float scale) {
  pdl_wait();
  pdl_trigger();
  constexpr int G = 4;                 // query heads per KV head
  constexpr int NW = 4;                // warps
  constexpr int SG = 16;               // slots per warp step
  constexpr int RB = HD * 2 + 16;      // padded row bytes (conflict-free ldmatrix)
  constexpr int STB = SG * RB;         // K (or V) bytes of one step
  constexpr int KS = HD / 16;          // k-steps of the scores
  constexpr int NB = HD / 8;           // n-blocks of the output
  static_assert(sizeof(KT) == 2, "fp16 cache");
  __shared__ __align__(16) float q[G][HD];
  __shared__ float kn_new[HD], vn_new[HD];
  __shared__ float wm[NW][G], wl[NW][G];
  __shared__ float red[8];
  extern __shared__ __align__(1024) unsigned char smraw[];
  const Dims& d = e.d;
  const int it = blockIdx.x;
  const int s = it % ns, g = (it / ns) % d.Hkv, b = it / (ns * d.Hkv);
  const int sid = e.bs[b].sid;
  float* outp = e.apart + static_cast<size_t>(it) * G * (HD + 2);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (stream_done(e, sid)) return;
  const int pos = ldcgi(&e.st[sid].pos);
  const int n = pos + 1;
  // the stream's own split count (a function of its context only, so that a stream's result does
  // not depend on the other streams of the batch); items beyond it stay empty
  const int nsb = min(ns, (n + kAttnChunk - 1) / kAttnChunk);
  const int chunk = (n + nsb - 1) / nsb;
  const int s0 = s * chunk, s1 = s < nsb ? min(n, s0 + chunk) : s0;
  if (s0 >= s1) {
    if (tid < G) {
      outp[G * HD + tid] = -INFINITY;
      outp[G * HD + G + tid] = 0.f;
    }
    return;
  }
  const int QKV = (d.Hq + 2 * d.Hkv) * HD;
  const int NC = e.nb;
  const bool has_new = pos >= s0 && pos < s1;
  const size_t slots = static_cast<size_t>(e.kv_slots);
  const size_t base = ((static_cast<size_t>(layer) * e.max_streams + sid) * d.Hkv + g) * slots * HD;
  KT* Kc = reinterpret_cast<KT*>(e.kc) + base;
  KT* Vc = reinterpret_cast<KT*>(e.vc) + base;
  // this warp's 16-slot groups: warp, warp + 4, ...
  const int ngrp = (s1 - s0 + SG - 1) / SG;
  const int nstep = ngrp > warp ? (ngrp - warp + NW - 1) / NW : 0;
  unsigned char* wst = smraw + static_cast<size_t>(warp) * kAttnStages * 2 * STB;
  auto stage = [&](int t) {
    if (t < nstep) {
      const int q0 = s0 + SG * (warp + NW * t);
      const int rows = min(SG, s1 - q0);
      unsigned char* dk = wst + (t % kAttnStages) * 2 * STB;
      constexpr int CPR = HD * 2 / 16;
      for (int c = lane; c < rows * CPR; c += 32) {
        const int r = c / CPR, cc = c % CPR;
        cp_async16(dk + r * RB + cc * 16, reinterpret_cast<const unsigned char*>(Kc + static_cast<size_t>(q0 + r) * HD) + cc * 16);
        cp_async16(dk + STB + r * RB + cc * 16,
                   reinterpret_cast<const unsigned char*>(Vc + static_cast<size_t>(q0 + r) * HD) + cc * 16);
      }
    }
    cp_async_commit();
  };
  // the old slots do not depend on this step: their copies start before the prologue
  for (int t = 0; t < kAttnStages - 1; ++t) stage(t);
  // q of the G heads (and the new k, v) from the split partials: all loads first
  {
    constexpr int PER = G * HD / 128;
    float a[PER];
#pragma unroll
    for (int u = 0; u < PER; ++u) a[u] = 0.f;
#pragma unroll 4
    for (int sp = 0; sp < splits; ++sp) {
      const float* pp = part + (static_cast<size_t>(sp) * NC + b) * QKV + (g * G) * HD;
#pragma unroll
      for (int u = 0; u < PER; ++u) a[u] += __ldcg(pp + tid + u * 128);
    }
#pragma unroll
    for (int u = 0; u < PER; ++u) (&q[0][0])[tid + u * 128] = a[u];
    if (has_new)
      for (int t = tid; t < HD; t += 128) {
        float kk = 0.f, vv = 0.f;
    #pragma unroll 4
    for (int sp = 0; sp < splits; ++sp) {
          const float* pp = part + (static_cast<size_t>(sp) * NC + b) * QKV;
          kk += __ldcg(pp + d.Hq * HD + g * HD + t);
          vv += __ldcg(pp + (d.Hq + d.Hkv) * HD + g * HD + t);
        }
        kn_new[t] = kk;
        vn_new[t] = vv;
      }
  }
  const float2* rrow = e.rope + static_cast<size_t>(pos) * (HD / 2);
  norm_rope_heads<HD>(&q[0][0], G, qn, d.qk_norm != 0, d.esz, d.eps, rrow, red);
  if (has_new) {
    norm_rope_heads<HD>(kn_new, 1, kn, d.qk_norm != 0, d.esz, d.eps, rrow, red);
    for (int t = tid; t < HD; t += 128) {
      const KT kq = tokv<KT>(kn_new[t]), vq = tokv<KT>(vn_new[t]);
      Kc[static_cast<size_t>(pos) * HD + t] = kq;
      Vc[static_cast<size_t>(pos) * HD + t] = vq;
      kn_new[t] = kvf<KT>(kq);
      vn_new[t] = kvf<KT>(vq);
    }
    __syncthreads();
  }
  // A fragments of the scaled queries: row gq = lane/4 (< 8: head gq & 3, hi or remainder part)
  const int gq = lane >> 2, tq = lane & 3, hq = gq & 3, partq = gq >> 2;
  uint32_t qa[KS][2];
#pragma unroll
  for (int ks = 0; ks < KS; ++ks) {
    const int e0 = 16 * ks + 2 * tq;
    qa[ks][0] = pack_h2(h_part(q[hq][e0] * scale, partq), h_part(q[hq][e0 + 1] * scale, partq));
    qa[ks][1] = pack_h2(h_part(q[hq][e0 + 8] * scale, partq), h_part(q[hq][e0 + 9] * scale, partq));
  }
  float o[NB][4];
#pragma unroll
  for (int nb = 0; nb < NB; ++nb) o[nb][0] = o[nb][1] = o[nb][2] = o[nb][3] = 0.f;
  float m_run = -INFINITY, l_run = 0.f;  // of head hq
  const int lr = lane & 7, lm = lane >> 3;  // ldmatrix: row within a matrix, matrix index
  for (int t = 0; t < nstep; ++t) {
    stage(t + kAttnStages - 1);
    cp_async_wait_group<kAttnStages - 1>();
    __syncwarp();
    const int q0 = s0 + SG * (warp + NW * t);
    const int rows = min(SG, s1 - q0);
    unsigned char* dk = wst + (t % kAttnStages) * 2 * STB;
    unsigned char* dv = dk + STB;
    if (has_new && pos >= q0 && pos < q0 + SG) {
      // the copy of the new slot may predate its store: use the values computed here
      KT* kr = reinterpret_cast<KT*>(dk + (pos - q0) * RB);
      KT* vr = reinterpret_cast<KT*>(dv + (pos - q0) * RB);
      for (int u = lane; u < HD; u += 32) {
        kr[u] = tokv<KT>(kn_new[u]);
        vr[u] = tokv<KT>(vn_new[u]);
      }
    }
    if (rows < SG) {
      // rows past the range: zero V (their probability is 0, and 0 * stale data must stay 0)
      for (int c = lane; c < (SG - rows) * (HD / 2); c += 32) {
        const int r = rows + c / (HD / 2), cc = c % (HD / 2);
        reinterpret_cast<uint32_t*>(dv + r * RB)[cc] = 0u;
        reinterpret_cast<uint32_t*>(dk + r * RB)[cc] = 0u;
      }
    }
    __syncwarp();
    // scores of the two 8-slot blocks
    float sc[2][4];
#pragma unroll
    for (int blk = 0; blk < 2; ++blk) {
      sc[blk][0] = sc[blk][1] = sc[blk][2] = sc[blk][3] = 0.f;
#pragma unroll
      for (int ks = 0; ks < KS; ks += 2) {
        uint32_t bf[4];
        // matrices: (slots blk*8.., e 16ks), (.., 16ks+8), (.., 16ks+16), (.., 16ks+24)
        ldsm_x4(smem_u32(dk + (blk * 8 + lr) * RB + (16 * ks + 8 * lm) * 2), bf);
        mma_f16(sc[blk], qa[ks][0], qa[ks][1], bf[0], bf[1]);
        mma_f16(sc[blk], qa[ks + 1][0], qa[ks + 1][1], bf[2], bf[3]);
      }
    }
    // full scores (hi + remainder rows), masked; lane holds head hq, slots blk*8 + 2tq + {0,1}
    float v[4];
#pragma unroll
    for (int blk = 0; blk < 2; ++blk)
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const float x = sc[blk][c] + __shfl_xor_sync(0xffffffffu, sc[blk][c], 16);
        v[blk * 2 + c] = (blk * 8 + 2 * tq + c < rows) ? x : -INFINITY;
      }
    float mt = fmaxf(fmaxf(v[0], v[1]), fmaxf(v[2], v[3]));
    mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 1));
    mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 2));
    const float mn = fmaxf(m_run, mt);
    const float cf = m_run == -INFINITY ? 0.f : expf(m_run - mn);
    float pv[4], ps = 0.f;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      pv[u] = v[u] == -INFINITY ? 0.f : expf(v[u] - mn);
      ps += pv[u];
    }
    ps += __shfl_xor_sync(0xffffffffu, ps, 1);
    ps += __shfl_xor_sync(0xffffffffu, ps, 2);
    l_run = l_run * cf + ps;
    m_run = mn;
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
      o[nb][0] *= cf;
      o[nb][1] *= cf;
    }
    // P as the A operand: row gq = head hq, hi (gq < 4) or remainder; k = slot of the group
    const uint32_t pa0 = pack_h2(h_part(pv[0], partq), h_part(pv[1], partq));
    const uint32_t pa2 = pack_h2(h_part(pv[2], partq), h_part(pv[3], partq));
#pragma unroll
    for (int nbp = 0; nbp < NB / 2; ++nbp) {
      uint32_t bf[4];
      // matrices: (slots 0-7, e 16nbp), (slots 8-15, e 16nbp), (slots 0-7, e 16nbp+8), (slots 8-15, ..)
      ldsm_x4_t(smem_u32(dv + ((lm & 1) * 8 + lr) * RB + (16 * nbp + 8 * (lm >> 1)) * 2), bf);
      mma_f16(o[2 * nbp], pa0, pa2, bf[0], bf[1]);
      mma_f16(o[2 * nbp + 1], pa0, pa2, bf[2], bf[3]);
    }
    __syncwarp();
  }
  cp_async_wait_group<0>();
  __syncwarp();
  // the warp's result (hi + remainder rows added) into its own staging area, then combined
  float* ow = reinterpret_cast<float*>(wst);
#pragma unroll
  for (int nb = 0; nb < NB; ++nb)
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const float x = o[nb][c] + __shfl_xor_sync(0xffffffffu, o[nb][c], 16);
      if (partq == 0) ow[hq * HD + nb * 8 + 2 * tq + c] = x;
    }
  if (lane < 16 && (lane & 3) == 0) {
    wm[warp][hq] = m_run;
    wl[warp][hq] = l_run;
  }
  __syncthreads();
  for (int t2 = tid; t2 < G * HD; t2 += 128) {
    const int h = t2 / HD;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, wm[w][h]);
    float acc = 0.f, l = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float cw = wm[w][h] == -INFINITY ? 0.f : expf(wm[w][h] - M);
      acc = fmaf(cw, reinterpret_cast<const float*>(smraw + static_cast<size_t>(w) * kAttnStages * 2 * STB)[t2], acc);
      l = fmaf(cw, wl[w][h], l);
    }
    outp[t2] = acc;
    if (t2 % HD == 0) {
      outp[G * HD + h] = M;
      outp[G * HD + G + h] = l;
    }
  }
}

// Prompt attention on the tensor cores (FlashAttention-style, causal, GQA with 4 query heads per
// KV head).  CTA = (block of 8 prompt positions, KV head); warp w owns positions 2w, 2w+1 of the
// block as one m16 tile: rows r < 8 -> first position, r >= 8 -> second; (r & 7) >> 2 selects the
// fp16 hi part / remainder of the scaled query and r & 3 the query head.  K/V tiles of 32 slots
// are staged by the CTA (cp.async, double-buffered, padded rows); scores and P·V use mma.sync
// fp16 -> fp32 as in the decode attention, with the hi and lo rows added at the end.
// QKV: [Tc][QD] with q normalised and rotated; K/V of slots < pos0 + Tc already in the cache.
template <int HD>
__global__ void __launch_bounds__(128) k_attn_prefill_tc(const float* __restrict__ QKV, int Tc, int pos0, int Hq, int Hkv,
                                                         const __half* __restrict__ Kc, const __half* __restrict__ Vc,
                                                         int slots, float scale, float* __restrict__ O) {
  constexpr int G = 4, TS = 32;
  constexpr int RB = HD * 2 + 16;
  constexpr int KS = HD / 16, NB = HD / 8;
  __shared__ __align__(16) unsigned char kv[2][2][TS * RB];  // [buffer][K, V]
  const int g = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
  const int t0 = blockIdx.x * 8 + 2 * warp;  // the warp's first position (chunk-local)
  const int QD = (Hq + 2 * Hkv) * HD;
  const int gq = lane >> 2, tq = lane & 3, hq = gq & 3, partq = gq >> 2;
  // A fragments of the warp's queries: row gq -> position t0, row gq + 8 -> position t0 + 1
  uint32_t qa[KS][4];
  {
    const int tA = min(t0, Tc - 1), tB = min(t0 + 1, Tc - 1);
    const float* qA = QKV + static_cast<size_t>(tA) * QD + (g * G + hq) * HD;
    const float* qB = QKV + static_cast<size_t>(tB) * QD + (g * G + hq) * HD;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      const int e0 = 16 * ks + 2 * tq;
      qa[ks][0] = pack_h2(h_part(qA[e0] * scale, partq), h_part(qA[e0 + 1] * scale, partq));
      qa[ks][1] = pack_h2(h_part(qB[e0] * scale, partq), h_part(qB[e0 + 1] * scale, partq));
      qa[ks][2] = pack_h2(h_part(qA[e0 + 8] * scale, partq), h_part(qA[e0 + 9] * scale, partq));
      qa[ks][3] = pack_h2(h_part(qB[e0 + 8] * scale, partq), h_part(qB[e0 + 9] * scale, partq));
    }
  }
  const int pA = pos0 + t0, pB = pos0 + t0 + 1;       // causal limits of the two rows
  const int last = min(pos0 + blockIdx.x * 8 + 7, pos0 + Tc - 1);  // the block's last position
  const int ntiles = (last + 1 + TS - 1) / TS;
  const __half* Kh = Kc + static_cast<size_t>(g) * slots * HD;
  const __half* Vh = Vc + static_cast<size_t>(g) * slots * HD;
  auto stage = [&](int buf, int tt) {
    const int s0 = tt * TS, rows = min(TS, last + 1 - s0);
    constexpr int CPR = HD * 2 / 16;
    for (int c = tid; c < rows * CPR; c += 128) {
      const int r = c / CPR, cc = c % CPR;
      cp_async16(&kv[buf][0][r * RB + cc * 16], reinterpret_cast<const unsigned char*>(Kh + static_cast<size_t>(s0 + r) * HD) + cc * 16);
      cp_async16(&kv[buf][1][r * RB + cc * 16], reinterpret_cast<const unsigned char*>(Vh + static_cast<size_t>(s0 + r) * HD) + cc * 16);
    }
    // rows past the block's last position: zero (masked scores, zero probabilities)
    for (int c = tid; c < (TS - rows) * (HD / 2); c += 128) {
      const int r = rows + c / (HD / 2), cc = c % (HD / 2);
      reinterpret_cast<uint32_t*>(&kv[buf][0][r * RB])[cc] = 0u;
      reinterpret_cast<uint32_t*>(&kv[buf][1][r * RB])[cc] = 0u;
    }
    cp_async_commit();
  };
  float o[NB][4];
#pragma unroll
  for (int nb = 0; nb < NB; ++nb) o[nb][0] = o[nb][1] = o[nb][2] = o[nb][3] = 0.f;
  float mA = -INFINITY, mB = -INFINITY, lA = 0.f, lB = 0.f;
  const int lr = lane & 7, lm = lane >> 3;
  stage(0, 0);
  for (int tt = 0; tt < ntiles; ++tt) {
    const int buf = tt & 1;
    if (tt + 1 < ntiles) {
      stage(buf ^ 1, tt + 1);
      cp_async_wait_group<1>();
    } else {
      cp_async_wait_group<0>();
    }
    __syncthreads();
    const unsigned char* dk = kv[buf][0];
    const unsigned char* dv = kv[buf][1];
    // scores of the 4 8-slot blocks
    float sc[4][4];
#pragma unroll
    for (int blk = 0; blk < 4; ++blk) {
      sc[blk][0] = sc[blk][1] = sc[blk][2] = sc[blk][3] = 0.f;
#pragma unroll
      for (int ks = 0; ks < KS; ks += 2) {
        uint32_t bf[4];
        ldsm_x4(smem_u32(dk + (blk * 8 + lr) * RB + (16 * ks + 8 * lm) * 2), bf);
        mma_f16x(sc[blk], qa[ks], bf[0], bf[1]);
        mma_f16x(sc[blk], qa[ks + 1], bf[2], bf[3]);
      }
    }
    const int s0 = tt * TS;
    float vA[8], vB[8];
#pragma unroll
    for (int blk = 0; blk < 4; ++blk)
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int slot = s0 + blk * 8 + 2 * tq + c;
        const float xa = sc[blk][c] + __shfl_xor_sync(0xffffffffu, sc[blk][c], 16);
        const float xb = sc[blk][2 + c] + __shfl_xor_sync(0xffffffffu, sc[blk][2 + c], 16);
        vA[blk * 2 + c] = slot <= pA ? xa : -INFINITY;
        vB[blk * 2 + c] = slot <= pB ? xb : -INFINITY;
      }
    float mtA = -INFINITY, mtB = -INFINITY;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      mtA = fmaxf(mtA, vA[u]);
      mtB = fmaxf(mtB, vB[u]);
    }
    mtA = fmaxf(mtA, __shfl_xor_sync(0xffffffffu, mtA, 1));
    mtA = fmaxf(mtA, __shfl_xor_sync(0xffffffffu, mtA, 2));
    mtB = fmaxf(mtB, __shfl_xor_sync(0xffffffffu, mtB, 1));
    mtB = fmaxf(mtB, __shfl_xor_sync(0xffffffffu, mtB, 2));
    const float mnA = fmaxf(mA, mtA), mnB = fmaxf(mB, mtB);
    const float cfA = mA == -INFINITY ? 0.f : expf(mA - mnA);
    const float cfB = mB == -INFINITY ? 0.f : expf(mB - mnB);
    float psA = 0.f, psB = 0.f;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      vA[u] = vA[u] == -INFINITY ? 0.f : expf(vA[u] - mnA);
      vB[u] = vB[u] == -INFINITY ? 0.f : expf(vB[u] - mnB);
      psA += vA[u];
      psB += vB[u];
    }
    psA += __shfl_xor_sync(0xffffffffu, psA, 1);
    psA += __shfl_xor_sync(0xffffffffu, psA, 2);
    psB += __shfl_xor_sync(0xffffffffu, psB, 1);
    psB += __shfl_xor_sync(0xffffffffu, psB, 2);
    // a row that has seen no slot yet keeps m = -inf (its probabilities are 0)
    lA = lA * cfA + psA;
    lB = lB * cfB + psB;
    mA = mnA;
    mB = mnB;
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
      o[nb][0] *= cfA;
      o[nb][1] *= cfA;
      o[nb][2] *= cfB;
      o[nb][3] *= cfB;
    }
    // P·V over the two 16-slot halves of the tile
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      uint32_t pa[4];
      pa[0] = pack_h2(h_part(vA[4 * j + 0], partq), h_part(vA[4 * j + 1], partq));
      pa[1] = pack_h2(h_part(vB[4 * j + 0], partq), h_part(vB[4 * j + 1], partq));
      pa[2] = pack_h2(h_part(vA[4 * j + 2], partq), h_part(vA[4 * j + 3], partq));
      pa[3] = pack_h2(h_part(vB[4 * j + 2], partq), h_part(vB[4 * j + 3], partq));
#pragma unroll
      for (int nbp = 0; nbp < NB / 2; ++nbp) {
        uint32_t bf[4];
        ldsm_x4_t(smem_u32(dv + (16 * j + (lm & 1) * 8 + lr) * RB + (16 * nbp + 8 * (lm >> 1)) * 2), bf);
        mma_f16x(o[2 * nbp], pa, bf[0], bf[1]);
        mma_f16x(o[2 * nbp + 1], pa, bf[2], bf[3]);
      }
    }
    __syncthreads();
  }
  // hi + remainder rows, normalised; lanes of the hi part write
  const float iA = 1.0f / lA, iB = 1.0f / lB;
#pragma unroll
  for (int nb = 0; nb < NB; ++nb)
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const float xa = o[nb][c] + __shfl_xor_sync(0xffffffffu, o[nb][c], 16);
      const float xb = o[nb][2 + c] + __shfl_xor_sync(0xffffffffu, o[nb][2 + c], 16);
      if (partq == 0) {
        const int e = nb * 8 + 2 * tq + c;
        if (t0 < Tc) O[static_cast<size_t>(t0) * Hq * HD + (g * G + hq) * HD + e] = xa * iA;
        if (t0 + 1 < Tc) O[static_cast<size_t>(t0 + 1) * Hq * HD + (g * G + hq) * HD + e] = xb * iB;
      }
    }
}

// combine the splits of each (stream, KV head): o = Σ_s e^{m_s - M} o_s / Σ_s e^{m_s - M} l_s,
// written as the planes of the out-projection input (query head h at columns h*HD..)
template <int HD>
__global__ void __launch_bounds__(256) k_attn_comb(const BEnv e, int ns) {
  pdl_wait();
  pdl_trigger();
  constexpr int G = 4;
  constexpr int EPT = G * HD / 256;
  __shared__ float wgt[kMaxSplitsAttn][G];
  __shared__ float inv[G];
  const Dims& d = e.d;
  const int b = blockIdx.x / d.Hkv, g = blockIdx.x % d.Hkv;
  if (stream_done(e, e.bs[b].sid)) return;
  const float* base = e.apart + static_cast<size_t>(blockIdx.x) * ns * G * (HD + 2);
  const int tid = threadIdx.x;
  if (tid < G) {
    // weights e^{m_s - M} per split of head tid, and 1 / Σ_s e^{m_s - M} l_s
    float M = -INFINITY;
    for (int s = 0; s < ns; ++s) M = fmaxf(M, __ldcg(base + static_cast<size_t>(s) * G * (HD + 2) + G * HD + tid));
    float den = 0.f;
    for (int s = 0; s < ns; ++s) {
      const float* ps = base + static_cast<size_t>(s) * G * (HD + 2);
      const float m = __ldcg(ps + G * HD + tid);
      const float w = m == -INFINITY ? 0.f : expf(m - M);
      wgt[s][tid] = w;
      den = fmaf(w, __ldcg(ps + G * HD + G + tid), den);
    }
    inv[tid] = 1.0f / den;
  }
  __syncthreads();
  float num[EPT];
#pragma unroll
  for (int u = 0; u < EPT; ++u) num[u] = 0.f;
  for (int s = 0; s < ns; ++s) {
    const float* ps = base + static_cast<size_t>(s) * G * (HD + 2);
#pragma unroll
    for (int u = 0; u < EPT; ++u) {
      const int t = tid + u * 256;
      const float w = wgt[s][t / HD];
      if (w != 0.f) num[u] = fmaf(w, __ldcg(ps + t), num[u]);
    }
  }
#pragma unroll
  for (int u = 0; u < EPT; ++u) {
    const int t = tid + u * 256, h = t / HD;
    store_hilo(e.pO, e.ldO, b, (g * G + h) * HD + (t % HD), num[u] * inv[h]);
  }
}

// Fast-AR: per (stream, KV head), the call's new positions in order: q/k norm, RoPE at the
// position, K/V into the stream's window, attention over positions 0..p (ch.06 §1-§4).  The
// window's earlier rows are staged in shared memory once.
template <int HD>
__global__ void __launch_bounds__(256) k_attn_fast(const BEnv e, int layer, const void* qn, const void* kn,
                                                   const float* __restrict__ part, int splits, int npos, int pos0,
                                                   float scale) {
  pdl_wait();
  pdl_trigger();
  constexpr int G = 4;
  constexpr int WMAX = 16;
  __shared__ __align__(16) float q[G][HD];
  __shared__ __align__(16) float kw[WMAX][HD];
  __shared__ __align__(16) float vw[WMAX][HD];
  __shared__ float sc[G][WMAX];
  __shared__ float red[8];
  const Dims& d = e.d;
  const int b = blockIdx.x / d.Hkvf, g = blockIdx.x % d.Hkvf;
  const int sid = e.bs[b].sid;
  if (stream_done(e, sid)) return;
  const int tid = threadIdx.x;
  const int QKV = (d.Hqf + 2 * d.Hkvf) * HD;
  const int NC = e.nb * npos;
  const size_t wl = static_cast<size_t>(d.Wf) * d.Hkvf * HD;  // one layer of the window
  float* Kw = e.bfk + (static_cast<size_t>(b) * d.Lf + layer) * wl;
  float* Vw = e.bfv + (static_cast<size_t>(b) * d.Lf + layer) * wl;
  for (int t = tid; t < pos0 * HD; t += 256) {
    const int r = t / HD, k = t % HD;
    kw[r][k] = __ldcg(Kw + (static_cast<size_t>(r) * d.Hkvf + g) * HD + k);
    vw[r][k] = __ldcg(Vw + (static_cast<size_t>(r) * d.Hkvf + g) * HD + k);
  }
  for (int j = 0; j < npos; ++j) {
    const int c = b * npos + j, p = pos0 + j;
    {
      // q of the G heads, then k and v: loads first
      constexpr int PER = G * HD / 256;
      float a[PER];
      float kk = 0.f, vv = 0.f;
#pragma unroll
      for (int u = 0; u < PER; ++u) a[u] = 0.f;
  #pragma unroll 4
    for (int sp = 0; sp < splits; ++sp) {
        const float* pp = part + (static_cast<size_t>(sp) * NC + c) * QKV;
#pragma unroll
        for (int u = 0; u < PER; ++u) a[u] += __ldcg(pp + (g * G) * HD + tid + u * 256);
        if (tid < HD) {
          kk += __ldcg(pp + d.Hqf * HD + g * HD + tid);
          vv += __ldcg(pp + (d.Hqf + d.Hkvf) * HD + g * HD + tid);
        }
      }
      __syncthreads();
#pragma unroll
      for (int u = 0; u < PER; ++u) (&q[0][0])[tid + u * 256] = a[u];
      if (tid < HD) {
        kw[p][tid] = kk;
        vw[p][tid] = vv;
      }
    }
    const float2* rrow = e.rope_f + static_cast<size_t>(p) * (HD / 2);
    norm_rope_heads<HD>(&q[0][0], G, qn, d.qk_norm != 0, d.esz, d.eps, rrow, red);
    norm_rope_heads<HD>(&kw[p][0], 1, kn, d.qk_norm != 0, d.esz, d.eps, rrow, red);
    if (tid < HD) {
      Kw[(static_cast<size_t>(p) * d.Hkvf + g) * HD + tid] = kw[p][tid];
      Vw[(static_cast<size_t>(p) * d.Hkvf + g) * HD + tid] = vw[p][tid];
    }
    // scores: 4 threads per (head, position), a quarter of the head dimension each
    {
      const int pr = tid >> 2, qtr = tid & 3;
      const int h = pr / WMAX, t = pr % WMAX;
      float a = 0.f;
      if (t <= p) {
#pragma unroll 8
        for (int k = qtr * (HD / 4); k < (qtr + 1) * (HD / 4); ++k) a = fmaf(q[h][k], kw[t][k], a);
      }
      a += __shfl_xor_sync(0xffffffffu, a, 1);
      a += __shfl_xor_sync(0xffffffffu, a, 2);
      if (qtr == 0 && h < G) sc[h][t] = t <= p ? a * scale : -INFINITY;
    }
    __syncthreads();
    if (tid < G) {
      float m = -INFINITY;
      for (int t = 0; t <= p; ++t) m = fmaxf(m, sc[tid][t]);
      float l = 0.f;
      for (int t = 0; t <= p; ++t) {
        sc[tid][t] = expf(sc[tid][t] - m);
        l += sc[tid][t];
      }
      red[tid] = 1.0f / l;
    }
    __syncthreads();
    for (int t2 = tid; t2 < G * HD; t2 += 256) {
      const int h = t2 / HD, k = t2 % HD;
      float a = 0.f;
      for (int t = 0; t <= p; ++t) a = fmaf(sc[h][t], vw[t][k], a);
      store_hilo(e.pO, e.ldO, c, (g * G + h) * HD + k, a * red[h]);
    }
  }
}

// =========================================================================================
// draws and bookkeeping (one CTA of 256 threads per stream)
// =========================================================================================

// dst[i] = Σ_s part[s][col][i] for i < n (n <= 16 * blockDim.x), loads batched per thread
__device__ void sum_partials(float* dst, const float* __restrict__ part, int splits, int NC, int col, int n) {
  constexpr int R = 16;
  float a[R];
#pragma unroll
  for (int r = 0; r < R; ++r) a[r] = 0.f;
  for (int s = 0; s < splits; s += 4) {
    float t[4][R];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float* ps = part + (static_cast<size_t>(s + j) * NC + col) * n;
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const int i = threadIdx.x + r * blockDim.x;
        t[j][r] = (s + j < splits && i < n) ? __ldcg(ps + i) : 0.f;
      }
    }
#pragma unroll
    for (int r = 0; r < R; ++r) a[r] = (((a[r] + t[0][r]) + t[1][r]) + t[2][r]) + t[3][r];
  }
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int i = threadIdx.x + r * blockDim.x;
    if (i < n) dst[i] = a[r];
  }
}

__device__ void copy_row(float* dst, const float* src, int n) {
  for (int i = threadIdx.x; i < n; i += blockDim.x) dst[i] = ldcg(src + i);
}

__device__ __forceinline__ int checked(const BEnv& e, int v, int hi) {
  if (v < 0 || v >= hi) {
    atomicCAS(&e.ctl->error, 0, S2_EINVAL);
    return 0;
  }
  return v;
}

// main draw, repetition-aware redraw, clamp, stop (ch.06 §5, §6); then the planes of the stream's
// hidden state for fast_project_in
__global__ void __launch_bounds__(kConsumers) k_samp_main(const BEnv e) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ __align__(1024) unsigned char smraw[];
  SampScratch& W = *reinterpret_cast<SampScratch*>(smraw);
  __shared__ int flag;
  const Dims& d = e.d;
  const int b = blockIdx.x;
  const BStream& bs = e.bs[b];
  const int sid = bs.sid;
  StreamState* st = e.st + sid;
  if (stream_done(e, sid)) return;
  const int f = frame_index(e);
  const float* lg = e.logits + static_cast<size_t>(sid) * e.lstride;
  const float* hid = e.hidden + static_cast<size_t>(sid) * d.D;
  if (bs.dbg_main) copy_row(bs.dbg_main + static_cast<size_t>(f) * d.A, lg, d.A);
  if (bs.dbg_hidden) copy_row(bs.dbg_hidden + static_cast<size_t>(f) * d.D, hid, d.D);
  const int fd = ldcgi(&st->frames_done);
  const float* E = bs.expo + static_cast<size_t>(f) * kDraws * kTopK;
  const bool block_end = fd < bs.min_tokens;
  // a stop request (s2_stop_stream) ends the stream at this frame boundary, like im_end
  if (threadIdx.x == 0) flag = ld_volatile_int(&st->stop_req);
  __syncthreads();
  if (flag) {
    if (threadIdx.x == 0) {
      st->done = 1;
      st->n_out = f;
    }
    return;
  }
  __syncthreads();
  int d0 = draw(d, W, lg, d.A, true, block_end, bs.T, bs.top_p, E);
  if (threadIdx.x == 0) {
    if (bs.dbg_draws) bs.dbg_draws[f * kDraws + 0] = d0;
    if (bs.forced) {
      d0 = bs.forced[f * kDraws + 0];
      if (d0 < 0 || d0 >= d.V) {
        atomicCAS(&e.ctl->error, 0, S2_EINVAL);
        d0 = d.im_end;
      }
    }
    flag = d0;
  }
  __syncthreads();
  d0 = flag;
  __syncthreads();
  if (d0 == d.im_end || d0 < 0) {
    if (threadIdx.x == 0) {
      st->done = 1;
      st->n_out = f;
      if (bs.dbg_draws)
        for (int k = 1; k < kDraws; ++k) bs.dbg_draws[f * kDraws + k] = -1;
    }
    return;
  }
  int d1 = draw(d, W, lg, d.A, true, block_end, bs.ras_T, bs.ras_top_p, E + kTopK);
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    if (lane == 0) {
      if (bs.dbg_draws) bs.dbg_draws[f * kDraws + 1] = d1;
      if (bs.forced) d1 = checked(e, bs.forced[f * kDraws + 1], d.V);
      if (d1 < 0) d1 = d0;
    }
    d1 = __shfl_sync(0xffffffffu, d1, 0);
    const int wl = ldcgi(&st->wlen);
    const int wv = lane < wl ? ldcgi(&st->window[lane]) : -1;
    const bool seen = __any_sync(0xffffffffu, lane < wl && wv == d0);
    const bool trig = seen && d0 >= d.sem_lo && d0 <= d.sem_hi;
    const int tok = trig ? d1 : d0;
    if (wl < bs.ras_window) {
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
      e.bfcode[b * 16 + 0] = code0;
      e.stage[(static_cast<size_t>(sid) * kMaxFramesPerCall + f) * d.ncb + 0] = code0;
      st->frames_done = fd + 1;
    }
  }
  for (int k = threadIdx.x; k < d.D; k += blockDim.x) store_hilo(e.pX, e.ldX, b, k, ldcg(hid + k));
}

// one Fast-AR draw (codebook cb) from the summed fast_output partials; then the next call's new
// input row (fast_embeddings[code], normalised with the first Fast-AR layer's attention norm),
// or after the last codebook the Slow-AR input embedding of the frame (normalised likewise)
__global__ void __launch_bounds__(kConsumers) k_samp_fast(const BEnv e, int cb, const float* part, int splits,
                                                          const void* an_fast0, const void* an_slow0) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ __align__(1024) unsigned char smraw[];
  SampScratch& W = *reinterpret_cast<SampScratch*>(smraw);
  __shared__ int flag;
  __shared__ float red[kConsumers / 32];
  const Dims& d = e.d;
  const int b = blockIdx.x;
  const BStream& bs = e.bs[b];
  const int sid = bs.sid;
  StreamState* st = e.st + sid;
  if (stream_done(e, sid)) return;
  const int f = frame_index(e);
  float* fl = e.bflog + static_cast<size_t>(b) * d.cbs;
  const int NC = e.nb;
  sum_partials(fl, part, splits, NC, b, d.cbs);
  // the draw copies the row into shared memory through L2 (cp.async): make the stores visible there
  __threadfence();
  __syncthreads();
  if (bs.dbg_fast) copy_row(bs.dbg_fast + (static_cast<size_t>(f) * (d.ncb - 1) + (cb - 1)) * d.cbs, fl, d.cbs);
  const float* E = bs.expo + static_cast<size_t>(f) * kDraws * kTopK + (1 + cb) * kTopK;
  int dc = draw(d, W, fl, d.cbs, false, false, bs.T, bs.top_p, E);
  if (threadIdx.x == 0) {
    if (bs.dbg_draws) bs.dbg_draws[f * kDraws + 1 + cb] = dc;
    if (bs.forced) dc = checked(e, bs.forced[f * kDraws + 1 + cb], d.cbs);
    if (dc < 0) dc = 0;
    e.bfcode[b * 16 + cb] = dc;
    st->vals[1 + cb] = dc;
    e.stage[(static_cast<size_t>(sid) * kMaxFramesPerCall + f) * d.ncb + cb] = dc;
    if (cb == d.ncb - 1) st->n_out = f + 1;
    flag = dc;
  }
  __syncthreads();
  dc = flag;
  // next input row, normalised, as planes at column b
  const bool slow = cb == d.ncb - 1;
  const int K = slow ? d.D : d.Df;
  const void* nw = slow ? an_slow0 : an_fast0;
  float* xr = slow ? e.bx + static_cast<size_t>(b) * d.D : e.bfx + static_cast<size_t>(b) * 2 * d.Df;
  int tok = 0;
  float msem = 0.f;
  if (slow) {
    tok = ldcgi(&st->vals[0]);
    msem = (tok >= d.sem_lo && tok <= d.sem_hi) ? 1.f : 0.f;
  }
  // the row in registers (K <= 12 * 256): codebook-outer accumulation keeps the loads in flight
  constexpr int RP = (kPrepMaxK + kConsumers - 1) / kConsumers;
  float v[RP];
#pragma unroll
  for (int i = 0; i < RP; ++i) v[i] = 0.f;
  if (slow) {
    // the frame's codes (this CTA drew them: its bfcode row), then every codebook row's loads
    // issued together; the sum keeps codebook order
    int codes[kMaxCodebooks];
#pragma unroll
    for (int c2 = 0; c2 < kMaxCodebooks; ++c2) codes[c2] = c2 < d.ncb ? (c2 == cb ? dc : e.bfcode[b * 16 + c2]) : 0;
#pragma unroll
    for (int c2 = 0; c2 < kMaxCodebooks; ++c2) {
      if (c2 >= d.ncb) break;
      const size_t row = (static_cast<size_t>(c2) * d.cbs + codes[c2]) * K;
#pragma unroll
      for (int i = 0; i < RP; ++i) {
        const int k = threadIdx.x + i * kConsumers;
        if (k < K) v[i] = __fadd_rn(v[i], wload(e.CE, row + k, d.esz));
      }
    }
#pragma unroll
    for (int i = 0; i < RP; ++i) {
      const int k = threadIdx.x + i * kConsumers;
      if (k < K)
        v[i] = __fadd_rn(__fmul_rn(d.sem_scale, wload(e.E, static_cast<size_t>(tok) * K + k, d.esz)), __fmul_rn(msem, v[i]));
    }
  } else {
#pragma unroll
    for (int i = 0; i < RP; ++i) {
      const int k = threadIdx.x + i * kConsumers;
      if (k < K) v[i] = wload(e.FE, static_cast<size_t>(dc) * K + k, d.esz);
    }
  }
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < RP; ++i) {
    const int k = threadIdx.x + i * kConsumers;
    if (k < K) {
      xr[k] = v[i];
      ss += v[i] * v[i];
    }
  }
  const float r = 1.0f / sqrtf(block_sum<kConsumers>(ss, red) / static_cast<float>(K) + d.eps);
#pragma unroll
  for (int i = 0; i < RP; ++i) {
    const int k = threadIdx.x + i * kConsumers;
    if (k < K) store_hilo(e.pX, e.ldX, b, k, (v[i] * r) * wload(nw, k, d.esz));
  }
}

// admissible Slow-AR logits of the step: the semantic rows from the partials, im_end by one dot
// product with the normalised hidden state; then the stream position advances
__global__ void __launch_bounds__(256) k_logits_fin(const BEnv e, const float* part, int splits) {
  pdl_wait();
  pdl_trigger();
  __shared__ float red[8];
  const Dims& d = e.d;
  const int b = blockIdx.x;
  const int sid = e.bs[b].sid;
  if (stream_done(e, sid)) return;
  float* lg = e.logits + static_cast<size_t>(sid) * e.lstride;
  const int NC = e.nb;
  sum_partials(lg, part, splits, NC, b, d.cbs);
  const float* h = e.hidden + static_cast<size_t>(sid) * d.D;
  float a = 0.f;
  for (int k = threadIdx.x; k < d.D; k += blockDim.x)
    a = fmaf(wload(e.E, static_cast<size_t>(d.im_end) * d.D + k, d.esz), ldcg(h + k), a);
  a = block_sum<256>(a, red);
  if (threadIdx.x == 0) {
    lg[d.cbs] = a;
    e.st[sid].pos = ldcgi(&e.st[sid].pos) + 1;
  }
}

__global__ void k_call_start(const BEnv e) {
  pdl_wait();
  pdl_trigger();
  const int b = threadIdx.x;
  if (b < e.nb) e.st[e.bs[b].sid].n_out = 0;
  if (b == 0) e.bctl[0] = 0;
}

__global__ void k_frame_end(const BEnv e) {
  pdl_wait();
  pdl_trigger();
  if (threadIdx.x == 0) e.bctl[0] = e.bctl[0] + 1;
}

}  // namespace

// =========================================================================================
// host side
// =========================================================================================

namespace {

int round16(int v) { return (v + 15) / 16 * 16; }

// dynamic shared memory of the Slow-AR attention: per warp, kAttnStages groups of 16 K and 16 V
// rows (padded)
constexpr int attn_smem(int hd) { return 4 * kAttnStages * 2 * 16 * (hd * 2 + 16); }

struct GemvPlan {
  int tiles, splits, per, atoms, nmat, M, K;
};

GemvPlan plan_gemv(int M, int K, int nmat, int sms, bool whole_k, int max_splits = 1 << 30, int atom = kAtom) {
  GemvPlan g{};
  g.M = M;
  g.K = K;
  g.nmat = nmat;
  g.atoms = K / atom;
  g.tiles = (M + kTileM - 1) / kTileM;
  int splits = whole_k ? 1 : std::max(1, std::min(std::min(g.atoms, max_splits), sms / std::max(1, g.tiles * nmat)));
  g.per = (g.atoms + splits - 1) / splits;
  g.splits = (g.atoms + g.per - 1) / g.per;
  return g;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 2-D bf16 tensor map over rows of `inner` elements (row pitch ld elements), box {64, box_rows},
// 128-byte swizzle
bool encode_map(CUtensorMap* m, const void* base, int inner, long long rows, int ld, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(kAtom), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D fp8 (byte) tensor map over rows x K codes, box {128, 128}, 128-byte swizzle
bool encode_map8(CUtensorMap* m, const void* base, int K, long long rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(K)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(kAtom8), static_cast<cuuint32_t>(kTileM)};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// fp8 projection launch shape: stages that fit the shared-memory budget (two CTAs per SM up to
// 128 MMA columns; wider tiles take one SM each, which also leaves their 512 TMEM columns alone)
constexpr int kGemv8WideBudget = 200 * 1024;
// weight-tile and planes stages that fit the budget (two CTAs per SM up to 128 MMA columns; wider
// tiles take one SM each, which also leaves their 512 TMEM columns alone)
int gemv8_smem(int N, int* nw, int* nb) {
  const int bstage = N * 256;
  const int budget = N <= 128 ? kGemvSmemBudget : kGemv8WideBudget;
  *nb = bstage < 16 * 1024 ? 3 : 2;
  *nw = std::min(kMaxGemvStages, (budget - *nb * bstage) / kA8Bytes);
  return std::max(kGemvSmemFloor, *nw * kA8Bytes + *nb * bstage + 1024 + static_cast<int>(sizeof(Gemv8Bars)));
}


}  // namespace

struct QEntry {
  CUtensorMap map;  // fp8 codes
  const float* s;   // row scales
};

struct Batch {
  BatchModel m;
  std::map<const void*, CUtensorMap> wmaps;
  std::map<const void*, QEntry> qmaps;  // bf16 weight -> its e4m3 copy (fp8 weight streaming)
  std::map<std::tuple<const void*, int, int>, CUtensorMap> pmaps;
  BatchSizes sz{};
  std::vector<BStream> host_bs;
  cudaStream_t cap = nullptr;   // private stream the frame is captured on
  // instantiated frame graphs by batch size: the per-call settings live in device memory, so a
  // graph serves every later call with the same number of streams
  std::map<int, cudaGraphExec_t> graphs;
};

bool batch_supported(const Dims& d, int max_streams, std::string* why) {
  auto no = [&](const char* w) {
    if (why) *why = w;
    return false;
  };
  if (d.wdt != S2_BF16 || d.kvdt != S2_F16) return no("batched decode needs bf16 weights and an fp16 KV cache");
  if (d.L == 0) return no("no Slow-AR");
  if (max_streams < 1 || max_streams > 64) return no("batched decode serves up to 64 streams per context");
  if (d.hd != 128 && d.hd != 64) return no("head_dim must be 64 or 128");
  if (d.Hq != 4 * d.Hkv || d.Hqf != 4 * d.Hkvf) return no("batched attention assumes 4 query heads per KV head");
  const int ks[6] = {d.D, d.Df, d.F, d.Ff, d.Hq * d.hd, d.Hqf * d.hdf};
  for (int k : ks)
    if (k % kAtom != 0) return no("projection lengths must be multiples of 64");
  if (d.D > kPrepMaxK || d.Df > kPrepMaxK) return no("model width above the column-preparation limit");
  if (d.Wf > 16) return no("Fast-AR window above 16");
  if (d.fp8)
    for (int k : ks)
      if (k % kAtom8 != 0) return no("fp8 projection lengths must be multiples of 128");
  return true;
}

BatchSizes batch_sizes(const Dims& d, int max_streams, int sms) {
  BatchSizes z{};
  const int ncmax = 2 * max_streams;
  z.planes_rows = static_cast<size_t>(round16(2 * ncmax));
  z.ldX = std::max(d.D, d.Df);
  z.ldO = std::max(d.Hq * d.hd, d.Hqf * d.hdf);
  z.ldH = std::max(d.F, d.Ff);
  const int QKV = (d.Hq + 2 * d.Hkv) * d.hd, QKVf = (d.Hqf + 2 * d.Hkvf) * d.hdf;
  size_t mx = 0;
  auto acc = [&](int M, int K, int nmat, bool whole, int nc) {
    const GemvPlan g = plan_gemv(M, K, nmat, kGemvCtasPerSm * sms, whole);
    mx = std::max(mx, static_cast<size_t>(g.nmat) * g.splits * nc * M);
  };
  acc(QKV, d.D, 1, false, max_streams);
  acc(d.D, d.Hq * d.hd, 1, false, max_streams);
  acc(d.F, d.D, 2, false, max_streams);
  acc(d.D, d.F, 1, false, max_streams);
  acc(d.cbs, d.D, 1, false, max_streams);
  acc(d.Df, d.D, 1, false, max_streams);
  acc(d.cbs, d.Df, 1, false, max_streams);
  acc(QKVf, d.Df, 1, false, ncmax);
  acc(d.Df, d.Hqf * d.hdf, 1, false, ncmax);
  acc(d.Ff, d.Df, 2, false, ncmax);
  acc(d.Df, d.Ff, 1, false, ncmax);
  z.part_floats = mx;
  z.apart_floats = static_cast<size_t>(max_streams) * d.Hkv * kMaxSplitsAttn * 4 * (d.hd + 2);
  return z;
}

size_t batch_stream_bytes(int max_streams) { return sizeof(BStream) * static_cast<size_t>(max_streams); }

Batch* batch_create(const BatchModel& m, std::string* err) {
  if (!encode_fn()) {
    *err = "cuTensorMapEncodeTiled is not available from the driver";
    return nullptr;
  }
  Batch* b = new Batch();
  b->m = m;
  b->sz = batch_sizes(m.d, m.max_streams, m.sms);
  const Dims& d = m.d;
  auto add = [&](const void* w, int rows, int cols) {
    CUtensorMap t;
    if (!encode_map(&t, w, cols, rows, cols, kTileM)) return false;
    b->wmaps[w] = t;
    return true;
  };
  bool ok = add(m.E, d.V, d.D) && add(m.FO, d.cbs, d.Df) && (!m.P || add(m.P, d.Df, d.D));
  const int QKV = (d.Hq + 2 * d.Hkv) * d.hd, QKVf = (d.Hqf + 2 * d.Hkvf) * d.hdf;
  for (int l = 0; l < d.L && ok; ++l) {
    const LayerW& w = m.slow[l];
    ok = add(w.wqkv, QKV, d.D) && add(w.wo, d.D, d.Hq * d.hd) && add(w.w1, d.F, d.D) && add(w.w3, d.F, d.D) &&
         add(w.w2, d.D, d.F);
  }
  for (int l = 0; l < d.Lf && ok; ++l) {
    const LayerW& w = m.fast[l];
    ok = add(w.wqkv, QKVf, d.Df) && add(w.wo, d.Df, d.Hqf * d.hdf) && add(w.w1, d.Ff, d.Df) &&
         add(w.w3, d.Ff, d.Df) && add(w.w2, d.Df, d.Ff);
  }
  for (int i = 0; i < m.n_qw && ok; ++i) {
    const QuantW& q = m.qw[i];
    QEntry e{};
    e.s = q.s;
    ok = encode_map8(&e.map, q.q, q.cols, q.rows);
    b->qmaps[q.w] = e;
  }
  if (!ok) {
    *err = "encoding a weight tensor map failed";
    delete b;
    return nullptr;
  }
  if (cudaStreamCreateWithFlags(&b->cap, cudaStreamNonBlocking) != cudaSuccess) {
    *err = "creating the capture stream failed";
    delete b;
    return nullptr;
  }
  if (cudaFuncSetAttribute(k_attn_slow<128, __half>, cudaFuncAttributeMaxDynamicSharedMemorySize, attn_smem(128)) !=
          cudaSuccess ||
      cudaFuncSetAttribute(k_attn_slow<64, __half>, cudaFuncAttributeMaxDynamicSharedMemorySize, attn_smem(64)) !=
          cudaSuccess) {
    *err = "setting the attention kernel's shared memory failed";
    delete b;
    return nullptr;
  }
  const int gsmem = kGemvSmemBudget + 1024 + static_cast<int>(sizeof(GemvBars));
  const int g8smem = kGemv8WideBudget + 1024 + static_cast<int>(sizeof(Gemv8Bars));
  if (cudaFuncSetAttribute(k_bgemv, cudaFuncAttributeMaxDynamicSharedMemorySize, gsmem) != cudaSuccess ||
      cudaFuncSetAttribute(k_bgemv8, cudaFuncAttributeMaxDynamicSharedMemorySize, g8smem) != cudaSuccess) {
    *err = "setting the projection kernel's shared memory failed";
    delete b;
    return nullptr;
  }
  return b;
}

int batch_prefill_proj(Batch* b, const void* w0, const void* w1, int M, int K, const uint16_t* planes, int ld, int NC,
                       float* part, void* stream) {
  if (NC < 1 || NC > kPrefillCols || K % kAtom != 0) return -1;
  const int N = round16(2 * NC);
  auto key = std::make_tuple(static_cast<const void*>(planes), N, K);
  auto it = b->pmaps.find(key);
  if (it == b->pmaps.end()) {
    CUtensorMap t;
    if (!encode_map(&t, planes, K, N, ld, N)) return -1;
    it = b->pmaps.emplace(key, t).first;
  }
  auto qa = b->qmaps.find(w0);
  if (qa != b->qmaps.end()) {
    auto qb = b->qmaps.find(w1 ? w1 : w0);
    if (qb == b->qmaps.end() || K % kAtom8 != 0) return -1;
    const GemvPlan g = plan_gemv(M, K, w1 ? 2 : 1, kGemvCtasPerSm * b->m.sms, false, 1 << 30, kAtom8);
    int nw = 0, nb = 0;
    const int smem = gemv8_smem(N, &nw, &nb);
    dim3 grid(g.tiles, g.splits, g.nmat);
    k_bgemv8<<<grid, kGemv8Threads, smem, static_cast<cudaStream_t>(stream)>>>(
        qa->second.map, qb->second.map, it->second, qa->second.s, qb->second.s, M, 0, N, NC, g.atoms, g.per, nw, nb,
        part, b->m.ctl);
    return cudaGetLastError() == cudaSuccess ? g.splits : -1;
  }
  const GemvPlan g = plan_gemv(M, K, w1 ? 2 : 1, kGemvCtasPerSm * b->m.sms, false);
  auto wa = b->wmaps.find(w0);
  auto wb = b->wmaps.find(w1 ? w1 : w0);
  if (wa == b->wmaps.end() || wb == b->wmaps.end()) return -1;
  const int sbytes = kABytes + N * 128;
  const int nst = std::min(kMaxGemvStages, kGemvSmemBudget / sbytes);
  const int smem = std::max(kGemvSmemFloor, nst * sbytes + 1024 + static_cast<int>(sizeof(GemvBars)));
  dim3 grid(g.tiles, g.splits, g.nmat);
  k_bgemv<<<grid, kGemvThreads, smem, static_cast<cudaStream_t>(stream)>>>(
      wa->second, wb->second, it->second, M, 0, N, NC, g.atoms, g.per, nst, part, b->m.ctl);
  return cudaGetLastError() == cudaSuccess ? g.splits : -1;
}

int batch_prefill_attn(const float* QKV, int Tc, int pos0, const Dims& d, const void* Kc, const void* Vc, int slots,
                       float scale, float* O, void* stream) {
  if (d.kvdt != S2_F16 || d.Hq != 4 * d.Hkv || (d.hd != 128 && d.hd != 64)) return -1;
  dim3 grid((Tc + 7) / 8, d.Hkv);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (d.hd == 128)
    k_attn_prefill_tc<128><<<grid, 128, 0, s>>>(QKV, Tc, pos0, d.Hq, d.Hkv, static_cast<const __half*>(Kc),
                                                 static_cast<const __half*>(Vc), slots, scale, O);
  else
    k_attn_prefill_tc<64><<<grid, 128, 0, s>>>(QKV, Tc, pos0, d.Hq, d.Hkv, static_cast<const __half*>(Kc),
                                                static_cast<const __half*>(Vc), slots, scale, O);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

size_t batch_prefill_part_floats(const Dims& d, int sms) {
  const int QKV = (d.Hq + 2 * d.Hkv) * d.hd;
  size_t mx = 0;
  auto acc = [&](int M, int K, int nmat) {
    const GemvPlan g = plan_gemv(M, K, nmat, kGemvCtasPerSm * sms, false);
    mx = std::max(mx, static_cast<size_t>(g.nmat) * g.splits * kPrefillCols * M);
  };
  acc(QKV, d.D, 1);
  acc(d.D, d.Hq * d.hd, 1);
  acc(d.F, d.D, 2);
  acc(d.D, d.F, 1);
  return mx;
}

int quantize_e4m3(const void* w, long long rows, int K, uint8_t* q, float* scales, void* stream) {
  if (rows <= 0 || K <= 0) return 0;
  const int grid = static_cast<int>(std::min<long long>(rows, 152LL * 8));
  k_quant_e4m3<<<grid, kQuantThreads, 0, static_cast<cudaStream_t>(stream)>>>(static_cast<const uint16_t*>(w), rows,
                                                                             K, q, scales);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

int e4m3_selfcheck(int* bad, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(bad, 0, sizeof(int), s) != cudaSuccess) return -1;
  k_e4m3_selfcheck<<<1, 256, 0, s>>>(bad);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

void batch_destroy(Batch* b) {
  if (!b) return;
  for (auto& kv : b->graphs) cudaGraphExecDestroy(kv.second);
  if (b->cap) cudaStreamDestroy(b->cap);
  delete b;
}

namespace {

struct Frame {
  Batch* b;
  BEnv e;
  cudaStream_t s;
  int nb;
  int ns;
  bool ok = true;

  // every kernel of the frame may start while its predecessor finishes (programmatic dependent
  // launch): each one waits for its predecessor's results in pdl_wait before using them
  template <typename... Exp, typename... Act>
  void launch(void (*k)(Exp...), dim3 grid, dim3 block, size_t smem, Act&&... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, k, std::forward<Act>(args)...) != cudaSuccess) ok = false;
  }

  const CUtensorMap& planes(uint16_t* buf, int N, int K, int ld) {
    auto key = std::make_tuple(static_cast<const void*>(buf), N, K);
    auto it = b->pmaps.find(key);
    if (it != b->pmaps.end()) return it->second;
    CUtensorMap t;
    if (!encode_map(&t, buf, K, N, ld, N)) ok = false;
    return b->pmaps[key] = t;
  }

  // projection of NC columns; returns the plan (partials layout)
  GemvPlan gemv(const void* w0, const void* w1, int M, int K, int row0, uint16_t* pl, int ld, int NC, bool whole_k,
               int max_splits = 1 << 30) {
    auto q0 = b->qmaps.find(w0);
    if (q0 != b->qmaps.end()) {
      const QEntry& qa = q0->second;
      const QEntry& qb = w1 ? b->qmaps.at(w1) : qa;
      const GemvPlan g = plan_gemv(M, K, w1 ? 2 : 1, kGemvCtasPerSm * b->m.sms, whole_k, max_splits, kAtom8);
      const int N = round16(2 * NC);
      const CUtensorMap& tb = planes(pl, N, K, ld);
      int nw = 0, nb = 0;
      const int smem = gemv8_smem(N, &nw, &nb);
      dim3 grid(g.tiles, g.splits, g.nmat);
      launch(k_bgemv8, grid, kGemv8Threads, smem, qa.map, qb.map, tb, qa.s, qb.s, M, row0, N, NC, g.atoms, g.per, nw, nb,
             e.part, e.ctl);
      return g;
    }
    const GemvPlan g = plan_gemv(M, K, w1 ? 2 : 1, kGemvCtasPerSm * b->m.sms, whole_k, max_splits);
    const int N = round16(2 * NC);
    const CUtensorMap& ta = b->wmaps.at(w0);
    const CUtensorMap& ta2 = w1 ? b->wmaps.at(w1) : ta;
    const CUtensorMap& tb = planes(pl, N, K, ld);
    const int sbytes = kABytes + N * 128;
    const int nst = std::min(kMaxGemvStages, kGemvSmemBudget / sbytes);
    const int smem = std::max(kGemvSmemFloor, nst * sbytes + 1024 + static_cast<int>(sizeof(GemvBars)));
    dim3 grid(g.tiles, g.splits, g.nmat);
    launch(k_bgemv, grid, kGemvThreads, smem, ta, ta2, tb, M, row0, N, NC, g.atoms, g.per, nst, e.part, e.ctl);
    return g;
  }

  void colprep(const ColPrep& p, int NC) { launch(k_colprep, NC, kPrepThreads, 0, e, p); }

  void run() {
    const Dims& d = e.d;
    const BatchModel& m = b->m;
    const size_t samp = sizeof(SampScratch);
    launch(k_samp_main, nb, kConsumers, samp, e);
    // Fast-AR call 1: positions 0 (projected hidden) and 1 (fast_embeddings[code_0])
    {
      ColPrep p{};
      p.npos = 2;
      p.K = d.Df;
      p.x = e.bfx;
      p.xb = 2 * d.Df;
      p.normw = m.fast[0].an;
      p.code_idx = 0;
      p.mode[1] = CM_FEROW;
      if (m.P) {
        const GemvPlan g = gemv(m.P, nullptr, d.Df, d.D, 0, e.pX, e.ldX, nb, false);
        p.mode[0] = CM_STORE;
        p.part = e.part;
        p.splits = g.splits;
        p.part_nc = nb;
        p.part_by_stream = 1;
      } else {
        p.mode[0] = CM_HIDDEN;
      }
      colprep(p, 2 * nb);
    }
    const float fscale = 1.0f / std::sqrt(static_cast<float>(d.hdf));
    const int QKVf = (d.Hqf + 2 * d.Hkvf) * d.hdf;
    for (int cb = 1; cb < d.ncb; ++cb) {
      const int npos = cb == 1 ? 2 : 1, pos0 = cb == 1 ? 0 : cb, NC = nb * npos;
      for (int l = 0; l < d.Lf; ++l) {
        const LayerW& w = m.fast[l];
        GemvPlan g = gemv(w.wqkv, nullptr, QKVf, d.Df, 0, e.pX, e.ldX, NC, false);
        if (d.hdf == 128)
          launch(k_attn_fast<128>, nb * d.Hkvf, 256, 0, e, l, w.qn, w.kn, e.part, g.splits, npos, pos0, fscale);
        else
          launch(k_attn_fast<64>, nb * d.Hkvf, 256, 0, e, l, w.qn, w.kn, e.part, g.splits, npos, pos0, fscale);
        g = gemv(w.wo, nullptr, d.Df, d.Hqf * d.hdf, 0, e.pO, e.ldO, NC, false);
        ColPrep p{};
        p.npos = npos;
        p.mode[0] = p.mode[1] = CM_RESID;
        p.K = d.Df;
        p.part = e.part;
        p.splits = g.splits;
        p.part_nc = NC;
        p.x = e.bfx;
        p.xb = 2 * d.Df;
        p.normw = w.fn;
        colprep(p, NC);
        g = gemv(w.w1, w.w3, d.Ff, d.Df, 0, e.pX, e.ldX, NC, false);
        launch(k_swiglu, dim3((d.Ff + 255) / 256, NC), 256, 0, e, e.part, d.Ff, NC, g.splits);
        g = gemv(w.w2, nullptr, d.Df, d.Ff, 0, e.pH, e.ldH, NC, false);
        p.splits = g.splits;
        const bool last = l == d.Lf - 1;
        p.normw = last ? m.fnorm : m.fast[l + 1].an;
        p.last_only = last ? 1 : 0;
        colprep(p, NC);
      }
      // its partials are summed by one CTA per stream: few splits
      const GemvPlan g = gemv(m.FO, nullptr, d.cbs, d.Df, 0, e.pX, e.ldX, nb, false, kSamplerSplits);
      launch(k_samp_fast, nb, kConsumers, samp, e, cb, e.part, g.splits, m.fast[0].an, m.slow[0].an);
    }
    // Slow-AR step
    const float sscale = 1.0f / std::sqrt(static_cast<float>(d.hd));
    const int QKV = (d.Hq + 2 * d.Hkv) * d.hd;
    for (int l = 0; l < d.L; ++l) {
      const LayerW& w = m.slow[l];
      GemvPlan g = gemv(w.wqkv, nullptr, QKV, d.D, 0, e.pX, e.ldX, nb, false);
      if (d.hd == 128) {
        launch(k_attn_slow<128, __half>, nb * d.Hkv * ns, 128, attn_smem(128), e, l, w.qn, w.kn, e.part, g.splits, ns,
                                                                             sscale);
        launch(k_attn_comb<128>, nb * d.Hkv, 256, 0, e, ns);
      } else {
        launch(k_attn_slow<64, __half>, nb * d.Hkv * ns, 128, attn_smem(64), e, l, w.qn, w.kn, e.part, g.splits, ns,
                                                                           sscale);
        launch(k_attn_comb<64>, nb * d.Hkv, 256, 0, e, ns);
      }
      g = gemv(w.wo, nullptr, d.D, d.Hq * d.hd, 0, e.pO, e.ldO, nb, false);
      ColPrep p{};
      p.npos = 1;
      p.mode[0] = p.mode[1] = CM_RESID;
      p.K = d.D;
      p.part = e.part;
      p.splits = g.splits;
      p.part_nc = nb;
      p.x = e.bx;
      p.xb = d.D;
      p.normw = w.fn;
      colprep(p, nb);
      g = gemv(w.w1, w.w3, d.F, d.D, 0, e.pX, e.ldX, nb, false);
      launch(k_swiglu, dim3((d.F + 255) / 256, nb), 256, 0, e, e.part, d.F, nb, g.splits);
      g = gemv(w.w2, nullptr, d.D, d.F, 0, e.pH, e.ldH, nb, false);
      p.splits = g.splits;
      const bool last = l == d.L - 1;
      p.normw = last ? m.norm : m.slow[l + 1].an;
      p.hid_out = last ? e.hidden : nullptr;
      colprep(p, nb);
    }
    const GemvPlan g = gemv(m.E, nullptr, d.cbs, d.D, d.sem_lo, e.pX, e.ldX, nb, false, kSamplerSplits);
    launch(k_logits_fin, nb, 256, 0, e, e.part, g.splits);
    launch(k_frame_end, 1, 32, 0, e);
  }
};

}  // namespace

int batch_decode(Batch* b, int n, const int* ids, int n_frames, const s2_sampling* params, const float* expo,
                 const int32_t* forced, const s2_debug_taps* taps, int max_ctx, void* stream, std::string* err) {
  const BatchModel& m = b->m;
  const Dims& d = m.d;
  if (n < 1 || n > m.max_streams) {
    *err = "batched decode: stream count out of range";
    return S2_EINVAL;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  b->host_bs.assign(n, BStream{});
  for (int k = 0; k < n; ++k) {
    BStream& t = b->host_bs[k];
    const size_t fo = static_cast<size_t>(k) * n_frames;
    const s2_sampling& p = params[k];
    t.sid = ids[k];
    t.min_tokens = p.min_tokens_before_end;
    t.ras_window = p.ras_window;
    t.T = p.temperature;
    t.top_p = p.top_p;
    t.ras_T = p.ras_temperature;
    t.ras_top_p = p.ras_top_p;
    t.expo = expo + fo * kDraws * kTopK;
    t.forced = forced ? forced + fo * kDraws : nullptr;
    if (taps) {
      t.dbg_main = taps->main_logits ? taps->main_logits + fo * d.A : nullptr;
      t.dbg_fast = taps->fast_logits ? taps->fast_logits + fo * (d.ncb - 1) * d.cbs : nullptr;
      t.dbg_hidden = taps->hidden ? taps->hidden + fo * d.D : nullptr;
      t.dbg_draws = taps->draws ? taps->draws + fo * kDraws : nullptr;
    }
  }
  if (cudaMemcpyAsync(m.bstreams, b->host_bs.data(), sizeof(BStream) * n, cudaMemcpyHostToDevice, s) != cudaSuccess) {
    *err = "copying the call settings failed";
    return S2_ECUDA;
  }
  Frame fr{};
  fr.b = b;
  fr.s = b->cap;
  fr.nb = n;
  (void)max_ctx;
  // attention items per (stream, KV head): enough for the longest context the KV slots allow, so
  // that one graph per stream count serves every call; each stream uses its context's share
  fr.ns = std::max(1, std::min(kMaxSplitsAttn, (m.kv_slots + kAttnChunk - 1) / kAttnChunk));
  BEnv& e = fr.e;
  e.d = d;
  e.nb = n;
  e.max_streams = m.max_streams;
  e.kv_slots = m.kv_slots;
  e.lstride = m.lstride;
  e.st = m.st;
  e.bs = static_cast<const BStream*>(m.bstreams);
  e.bctl = m.bctl;
  e.hidden = m.hidden;
  e.logits = m.logits;
  e.stage = m.stage;
  e.ctl = m.ctl;
  e.kc = m.kc;
  e.vc = m.vc;
  e.rope = m.rope;
  e.rope_f = m.rope_f;
  e.E = m.E;
  e.CE = m.CE;
  e.FE = m.FE;
  e.pX = m.pX;
  e.pO = m.pO;
  e.pH = m.pH;
  e.ldX = b->sz.ldX;
  e.ldO = b->sz.ldO;
  e.ldH = b->sz.ldH;
  e.part = m.part;
  e.bx = m.bx;
  e.bfx = m.bfx;
  e.bfk = m.bfk;
  e.bfv = m.bfv;
  e.apart = m.apart;
  e.bflog = m.bflog;
  e.bfcode = m.bfcode;
  k_call_start<<<1, 64, 0, s>>>(e);
  if (cudaGetLastError() != cudaSuccess) {
    *err = "batched call start failed";
    return S2_ECUDA;
  }
  cudaGraphExec_t exec = nullptr;
  auto cached = b->graphs.find(n);
  if (cached != b->graphs.end()) {
    exec = cached->second;
  } else {
    cudaGraph_t graph = nullptr;
    if (cudaStreamBeginCapture(b->cap, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
      *err = "graph capture could not begin";
      return S2_ECUDA;
    }
    fr.run();
    const cudaError_t ce = cudaStreamEndCapture(b->cap, &graph);
    if (ce != cudaSuccess || !fr.ok) {
      if (graph) cudaGraphDestroy(graph);
      *err = std::string("capturing the frame failed: ") + (fr.ok ? cudaGetErrorString(ce) : "launch or tensor map");
      return S2_ECUDA;
    }
    const cudaError_t ie = cudaGraphInstantiate(&exec, graph, 0);
    cudaGraphDestroy(graph);
    if (ie != cudaSuccess) {
      *err = "instantiating the frame graph failed";
      return S2_ECUDA;
    }
    b->graphs[n] = exec;
  }
  cudaError_t le = cudaSuccess;
  for (int f = 0; f < n_frames && le == cudaSuccess; ++f) le = cudaGraphLaunch(exec, s);
  if (le != cudaSuccess) {
    *err = std::string("launching the frame graph failed: ") + cudaGetErrorString(le);
    return S2_ECUDA;
  }
  return S2_OK;
}

}  // namespace s2
