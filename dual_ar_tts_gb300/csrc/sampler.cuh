// The draw of the S2-Pro sampler for one logits vector, shared by the persistent frame kernel and
// the batched decode kernels: 256 threads (named barrier 1) of one CTA.
#pragma once

#include <cstdint>

#include "ptx.cuh"
#include "s2_internal.h"

namespace s2 {
namespace {

// =========================================================================
// sampler (CTA 0): top-30 by (value desc, id asc), softmax, top-p (keep rank r iff r == 0 or
// Σ_{s<r} π_s < p), winner = argmax π_r / E_r (ties -> lower rank)
// =========================================================================

constexpr int kSampPer = 17;  // values per thread: 256 * 17 >= 4097

// id of entry i of a logits vector: main (admissible) -> token id; fast -> code
__device__ __forceinline__ int entry_id(const Dims& d, bool main, int i) {
  return main ? (i < d.cbs ? d.sem_lo + i : d.im_end) : i;
}

// total order of candidates: larger value first, equal values -> lower id first
__device__ __forceinline__ bool better_k(uint32_t ka, int ia, uint32_t kb, int ib) {
  return ka > kb || (ka == kb && ia < ib);
}

// order-preserving map of a float to an unsigned key (finite values map above 0x007fffff)
__device__ __forceinline__ uint32_t fkey(float z) {
  const uint32_t u = __float_as_uint(z);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float fval(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Sampler scratch in shared memory (256 consumer threads; kSampPer logits per thread).
constexpr int kSampHist = 4096;  // first-level histogram of the fallback selection: top 12 key bits
constexpr int kSampCand = 64;    // candidates the threshold selection ranks directly
struct SampScratch {
  int nvalid, cut, rem, nA, nB, result, pad[2];
  uint32_t thr, pad2[3];
  int wsum[kConsumerWarps];
  uint32_t aK[32];  // fallback: candidates above the boundary bin (fewer than 30)
  int aI[32];
  uint32_t bK[kSampCand];  // threshold selection: the candidates; fallback: the boundary bin
  int bI[kSampCand];
  uint32_t cK[32];  // the final candidates in rank order
  int cI[32];
  alignas(16) uint32_t mx[kConsumers];  // per-thread maximum keys
  int hist[kSampHist];
  alignas(16) uint32_t keys[kSampPer * kConsumers];  // fallback: the keys by entry index
};

// bitonic sort of 32 (key, id) pairs across a warp, one per lane: best (larger key, then lower
// id) first
__device__ __forceinline__ void warp_sort32(uint32_t& k, int& id) {
  const int lane = threadIdx.x & 31;
#pragma unroll 1
  for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll 1
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const uint32_t pk = __shfl_xor_sync(0xffffffffu, k, stride);
      const int pi = __shfl_xor_sync(0xffffffffu, id, stride);
      const bool lower = (lane & stride) == 0;
      const bool asc = (lane & size) == 0;  // "ascending" = best first
      if ((lower == asc) == better_k(pk, pi, k, id)) {
        k = pk;
        id = pi;
      }
    }
  }
}

// The kk-th largest of the 256 per-thread maxima W.mx, by one warp: bitonic sort of the 256 keys,
// 8 per lane (element e = 8·lane + j), largest first.  Strides 1-4 stay in a lane's registers,
// strides 8-128 pair lanes (lane ^ stride/8).
__device__ __forceinline__ uint32_t kth_of_maxima(const SampScratch& W, int kk) {
  const int lane = threadIdx.x & 31;
  uint32_t v[8];
  {
    const uint4 a = *reinterpret_cast<const uint4*>(&W.mx[8 * lane]);
    const uint4 b = *reinterpret_cast<const uint4*>(&W.mx[8 * lane + 4]);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  }
#pragma unroll
  for (int size = 2; size <= 256; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      if (stride < 8) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (j & stride) continue;
          // descending block iff bit `size` of the element index is 0
          const bool desc = size < 8 ? (j & size) == 0 : ((8 * lane) & size) == 0;
          const uint32_t a = v[j], b = v[j | stride];
          const uint32_t hi = max(a, b), lo = min(a, b);
          v[j] = desc ? hi : lo;
          v[j | stride] = desc ? lo : hi;
        }
      } else {
        const int ls = stride >> 3;
        const bool lower = (lane & ls) == 0;
        const bool desc = (lane & (size >> 3)) == 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint32_t p = __shfl_xor_sync(0xffffffffu, v[j], ls);
          v[j] = (lower == desc) ? max(v[j], p) : min(v[j], p);
        }
      }
    }
  }
  const int e = kk - 1, jj = e & 7;
  uint32_t r = v[0];
#pragma unroll
  for (int j = 1; j < 8; ++j)
    if (j == jj) r = v[j];
  return __shfl_sync(0xffffffffu, r, e >> 3);
}

// Fallback selection of the top kk (any tie pattern): the keys are in W.keys.  A 4096-bin histogram
// of the top 12 bits locates the bin holding the kk-th key; while that bin holds more than 64
// keys it is refined by the next 10 bits (at most twice).  Keys above the boundary and the boundary
// bin's keys are then sorted by two warps; more than 64 equal keys at full resolution are taken in
// id order one by one.  Writes W.cK / W.cI[0 .. kk) in rank order.
__device__ __noinline__ void select_hist(const Dims& d, SampScratch& W, bool main, int kk) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
#pragma unroll 1
  for (int b = tid; b < kSampHist; b += kConsumers) W.hist[b] = 0;
  if (tid == 0) {
    W.nA = 0;
    W.nB = 0;
  }
  named_bar(1, kConsumers);

  // ---- locate the kk-th largest key: prefix `pre` of its top (32 - shift) bits, `need` of the
  // keys with that prefix belong to the top kk
  uint32_t pre = 0u;
  int shift = 32, need = kk, n_eq = 0;
#pragma unroll 1
  for (int level = 0; level < 3; ++level) {
    const int width = level == 0 ? 12 : 10;
    const uint32_t prev = pre;
    shift -= width;
    const uint32_t mask = (1u << width) - 1u;
#pragma unroll 1
    for (int k = 0; k < kSampPer; ++k) {
      const uint32_t key = W.keys[k * kConsumers + tid];
      if (key && (level == 0 || (key >> (shift + width)) == prev)) atomicAdd(&W.hist[(key >> shift) & mask], 1);
    }
    named_bar(1, kConsumers);
    // bins from the top: thread t owns bins nb-1-t*per .. nb-per-t*per
    const int nb = 1 << width, per = nb / kConsumers;
    int c = 0;
#pragma unroll 4
    for (int j = 0; j < per; ++j) c += W.hist[nb - 1 - tid * per - j];
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    if (lane == 31) W.wsum[warp] = incl;
    named_bar(1, kConsumers);
    int before = incl - c;
#pragma unroll 1
    for (int w = 0; w < warp; ++w) before += W.wsum[w];
    if (before < need && before + c >= need) {
      int cum = before;
#pragma unroll 1
      for (int j = 0; j < per; ++j) {
        const int bin = nb - 1 - tid * per - j;
        const int h = W.hist[bin];
        if (cum + h >= need) {
          W.cut = bin;
          W.rem = need - cum;
          break;
        }
        cum += h;
      }
    }
    named_bar(1, kConsumers);
    const int cut = W.cut;
    need = W.rem;
    n_eq = W.hist[cut];
    pre = (prev << width) | static_cast<uint32_t>(cut);
    if (n_eq <= 64 || level == 2) break;
    named_bar(1, kConsumers);  // everyone has read the histogram
#pragma unroll 1
    for (int b = tid; b < 1024; b += kConsumers) W.hist[b] = 0;
    named_bar(1, kConsumers);
  }

  // ---- gather: keys above the boundary prefix (all in the top kk) and keys at it
#pragma unroll 1
  for (int k = 0; k < kSampPer; ++k) {
    const uint32_t key = W.keys[k * kConsumers + tid];
    if (!key) continue;
    const uint32_t hi = key >> shift;
    if (hi < pre) continue;
    const int id = entry_id(d, main, tid + k * kConsumers);
    if (hi > pre) {
      const int slot = atomicAdd(&W.nA, 1);
      W.aK[slot] = key;
      W.aI[slot] = id;
    } else {
      const int slot = atomicAdd(&W.nB, 1);
      if (slot < 64) {
        W.bK[slot] = key;
        W.bI[slot] = id;
      }
    }
  }
  named_bar(1, kConsumers);
  const int nA = W.nA;  // == kk - need
  if (warp == 0) {
    uint32_t k0 = lane < nA ? W.aK[lane] : 0u;
    int i0 = lane < nA ? W.aI[lane] : (0x7fffffff - lane);
    warp_sort32(k0, i0);
    if (lane < nA) {
      W.cK[lane] = k0;
      W.cI[lane] = i0;
    }
  } else if (warp == 1 && n_eq <= 64) {
    // boundary bin: bitonic sort of up to 64 pairs, two per lane (lane, lane + 32)
    uint32_t ka = lane < n_eq ? W.bK[lane] : 0u, kb = lane + 32 < n_eq ? W.bK[lane + 32] : 0u;
    int ia = lane < n_eq ? W.bI[lane] : (0x7fffffff - lane), ib = lane + 32 < n_eq ? W.bI[lane + 32] : (0x7fffffdf - lane);
#pragma unroll 1
    for (int size = 2; size <= 64; size <<= 1) {
#pragma unroll 1
      for (int stride = size >> 1; stride > 0; stride >>= 1) {
        if (stride == 32) {
          if (better_k(kb, ib, ka, ia)) {
            const uint32_t tk = ka; ka = kb; kb = tk;
            const int ti = ia; ia = ib; ib = ti;
          }
          continue;
        }
        const uint32_t pka = __shfl_xor_sync(0xffffffffu, ka, stride), pkb = __shfl_xor_sync(0xffffffffu, kb, stride);
        const int pia = __shfl_xor_sync(0xffffffffu, ia, stride), pib = __shfl_xor_sync(0xffffffffu, ib, stride);
        const bool lower = (lane & stride) == 0;
        if ((lower == ((lane & size) == 0)) == better_k(pka, pia, ka, ia)) {
          ka = pka;
          ia = pia;
        }
        if ((lower == (((lane + 32) & size) == 0)) == better_k(pkb, pib, kb, ib)) {
          kb = pkb;
          ib = pib;
        }
      }
    }
    if (lane < need) {
      W.cK[nA + lane] = ka;
      W.cI[nA + lane] = ia;
    }
    if (lane + 32 < need) {
      W.cK[nA + lane + 32] = kb;
      W.cI[nA + lane + 32] = ib;
    }
  }
  if (n_eq > 64) {
    // more than 64 equal keys at full resolution: the `need` lowest ids among them, one by one
    int last = -1;
#pragma unroll 1
    for (int r = 0; r < need; ++r) {
      int best = 0x7fffffff;
#pragma unroll 1
      for (int k = 0; k < kSampPer; ++k) {
        const int id = entry_id(d, main, tid + k * kConsumers);
        const uint32_t key = W.keys[k * kConsumers + tid];
        if (key && (key >> shift) == pre && id > last && id < best) best = id;
      }
      best = warp_min_i(best);
      if (lane == 0) W.wsum[warp] = best;
      named_bar(1, kConsumers);
      int m = W.wsum[0];
#pragma unroll 1
      for (int w = 1; w < kConsumerWarps; ++w) m = min(m, W.wsum[w]);
      if (tid == 0) {
        W.cK[nA + r] = pre << shift;
        W.cI[nA + r] = m;
      }
      last = m;
      named_bar(1, kConsumers);
    }
  }
  named_bar(1, kConsumers);
}

// One draw: the top-30 candidates by (value desc, id asc), then, in rank order exactly as the
// method states: softmax over them, keep rank r iff r == 0 or Σ_{s<r} π_s < top_p, winner =
// argmax π_r / E_r (ties -> lower rank).  Returns the drawn id in every consumer thread; -1 if
// nothing is drawable.
// Selection: order-preserving 32-bit keys of z = logit / T, kSampPer per thread in registers.  At
// least kk of the 256 per-thread maxima are >= the kk-th largest of them (thr), so at least kk keys
// are, and every key of the top kk is >= thr: the keys >= thr hold the top kk, ranked by the same
// total order.  They are gathered (one shared-memory counter per warp) and, when at most 64, each
// is ranked by counting the candidates ahead of it; more than 64 (heavy ties) take the histogram
// selection above.
__device__ __noinline__ int draw(const Dims& d, SampScratch& W, const float* logits, int n, bool main, bool mask_end,
                                 float temperature, float top_p, const float* E) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // the rank-r variate, needed at the end, and this thread's logits (entries tid + 256 k) are
  // requested first, every load in flight together
  const float ev = (warp == 0 && lane < kTopK) ? ldcg(E + lane) : 1.f;
  uint32_t key[kSampPer];
#pragma unroll
  for (int k = 0; k < kSampPer; ++k) {
    const int i = tid + k * kConsumers;
    key[k] = i < n ? __float_as_uint(ldcg(logits + i)) : 0u;
  }
  uint32_t mx = 0u;
  int nv = 0;
#pragma unroll
  for (int k = 0; k < kSampPer; ++k) {
    const int i = tid + k * kConsumers;
    const float l = __uint_as_float(key[k]);
    uint32_t kv = 0u;
    if (i < n && !(mask_end && main && entry_id(d, main, i) == d.im_end) && isfinite(l)) {
      // + 0: -0 and +0 compare equal, so they share one key
      kv = fkey(l / temperature + 0.0f);
      ++nv;
    }
    key[k] = kv;
    mx = max(mx, kv);
  }
  nv = warp_sum_i(nv);
  if (lane == 0) W.wsum[warp] = nv;
  W.mx[tid] = mx;
  if (tid == 0) W.nB = 0;
  named_bar(1, kConsumers);
  int nvalid = 0;
#pragma unroll
  for (int w = 0; w < kConsumerWarps; ++w) nvalid += W.wsum[w];
  if (nvalid == 0) {
    named_bar(1, kConsumers);  // uniform: every thread saw the same count, and has read it
    return -1;
  }
  const int kk = min(kTopK, nvalid);
  if (warp == 0) {
    const uint32_t t = kth_of_maxima(W, kk);
    if (lane == 0) W.thr = t;
  }
  named_bar(1, kConsumers);
  // ---- gather the keys >= thr (key 0 = not drawable): warp-local slots, one counter per warp
  const uint32_t thr = max(W.thr, 1u);
  int c = 0;
#pragma unroll
  for (int k = 0; k < kSampPer; ++k) c += key[k] >= thr ? 1 : 0;
  int incl = c;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  int base = 0;
  if (lane == 31 && incl > 0) base = atomicAdd(&W.nB, incl);
  int slot = __shfl_sync(0xffffffffu, base, 31) + incl - c;
#pragma unroll
  for (int k = 0; k < kSampPer; ++k) {
    if (key[k] >= thr) {
      if (slot < kSampCand) {
        W.bK[slot] = key[k];
        W.bI[slot] = entry_id(d, main, tid + k * kConsumers);
      }
      ++slot;
    }
  }
  named_bar(1, kConsumers);
  const int nb = W.nB;  // >= kk
  if (nb <= kSampCand) {
    // rank of each candidate = the candidates ahead of it in (key desc, id asc); the top kk land
    // at their ranks
    if (tid < nb) {
      const uint32_t mk = W.bK[tid];
      const int mi = W.bI[tid];
      int rank = 0;
#pragma unroll 4
      for (int j = 0; j < nb; ++j) rank += better_k(W.bK[j], W.bI[j], mk, mi) ? 1 : 0;
      if (rank < kk) {
        W.cK[rank] = mk;
        W.cI[rank] = mi;
      }
    }
    named_bar(1, kConsumers);
  } else {
#pragma unroll
    for (int k = 0; k < kSampPer; ++k) W.keys[k * kConsumers + tid] = key[k];
    named_bar(1, kConsumers);  // every thread has read W.nB before the selection resets it
    select_hist(d, W, main, kk);
  }
  // ---- warp 0: the draw over the kk candidates, rank r = lane.  The sums, whose rounding depends
  // on the order, are taken in rank order (every lane runs the same sequence over shuffled values)
  if (warp == 0) {
    const float z = lane < kk ? fval(W.cK[lane]) : 0.f;
    const float zmax = __shfl_sync(0xffffffffu, z, 0);
    const float e = lane < kk ? expf(z - zmax) : 0.f;
    float sum = 0.f;
#pragma unroll
    for (int r = 0; r < kTopK; ++r) {
      const float er = __shfl_sync(0xffffffffu, e, r);
      if (r < kk) sum += er;
    }
    const float pi = e / sum;
    float cum = 0.f;
    int kept = 0;
    bool open = true;
#pragma unroll
    for (int r = 0; r < kTopK; ++r) {
      const float pr = __shfl_sync(0xffffffffu, pi, r);
      if (r < kk && open) {
        if (r == 0 || cum < top_p) kept = r + 1;
        else open = false;
        cum += pr;
      }
    }
    // winner = argmax_{r < kept} π_r / E_r, ties -> lower rank
    float q = lane < kept ? pi / ev : -INFINITY;
    int rq = lane;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float q2 = __shfl_xor_sync(0xffffffffu, q, o);
      const int r2 = __shfl_xor_sync(0xffffffffu, rq, o);
      if (q2 > q || (q2 == q && r2 < rq)) {
        q = q2;
        rq = r2;
      }
    }
    if (lane == 0) W.result = W.cI[rq];
  }
  named_bar(1, kConsumers);
  const int out = W.result;
  named_bar(1, kConsumers);
  return out;
}

}  // namespace
}  // namespace s2
