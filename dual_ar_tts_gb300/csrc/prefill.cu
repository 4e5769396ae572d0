// Prefill of one stream (chunked over positions), the RoPE tables and code compaction.
//
// Prefill runs the Slow-AR stack over the prompt positions ([ch.02 §3.1-§3.2] of s2.cpp
// analysis "Overall architecture and Dual-AR data flow"; chunked prefill per ch.02 §4), writing
// K/V for slots 0..T-1 and keeping the normalised hidden and admissible logits of the last
// position.  Projections here are CUDA-core fp32 tiled GEMMs; attention is causal over the KV
// cache with an online softmax.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>

#include "ptx.cuh"
#include "s2_internal.h"

namespace s2 {

namespace {

constexpr int kBlk = 256;

__device__ __forceinline__ float block_sum(float v, float* sh) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) sh[w] = v;
  __syncthreads();
  float t = 0.f;
  for (int i = 0; i < static_cast<int>(blockDim.x >> 5); ++i) t += sh[i];
  return t;
}

// x[t] = sem_scale·E[r0] + m·Σ_c CE[c·CBS + r_{c+1}], m = [r0 semantic]  (ch.02 §3.2)
__global__ void k_embed(const int32_t* tok, int T, Dims d, const void* E, const void* CE, float* X, int* err) {
  const int t = blockIdx.x;
  if (t >= T) return;
  const int C = d.ncb + 1;
  int r0 = tok[static_cast<size_t>(t) * C];
  if (r0 < 0 || r0 >= d.V) {
    if (threadIdx.x == 0) atomicCAS(err, 0, S2_EINVAL);
    r0 = 0;
  }
  const float m = (r0 >= d.sem_lo && r0 <= d.sem_hi) ? 1.f : 0.f;
  for (int e = threadIdx.x; e < d.D; e += blockDim.x) {
    float acc = 0.f;
    for (int c = 0; c < d.ncb; ++c) {
      int code = tok[static_cast<size_t>(t) * C + 1 + c];
      if (code < 0 || code >= d.cbs) {
        atomicCAS(err, 0, S2_EINVAL);
        code = 0;
      }
      acc = __fadd_rn(acc, wload(CE, (static_cast<size_t>(c) * d.cbs + code) * d.D + e, d.esz));
    }
    X[static_cast<size_t>(t) * d.D + e] =
        __fadd_rn(__fmul_rn(d.sem_scale, wload(E, static_cast<size_t>(r0) * d.D + e, d.esz)), __fmul_rn(m, acc));
  }
}

// H[t] = X[t] · 1/sqrt(mean(X[t]^2) + eps) · w
__global__ void k_rmsnorm(const float* X, int D, const void* w, int esz, float eps, float* H) {
  __shared__ float sh[32];
  const float* x = X + static_cast<size_t>(blockIdx.x) * D;
  float s = 0.f;
  for (int e = threadIdx.x; e < D; e += blockDim.x) s += x[e] * x[e];
  const float tot = block_sum(s, sh);
  const float r = 1.0f / sqrtf(tot / static_cast<float>(D) + eps);
  for (int e = threadIdx.x; e < D; e += blockDim.x)
    H[static_cast<size_t>(blockIdx.x) * D + e] = (x[e] * r) * wload(w, e, esz);
}

// Y[t][r] (=|+=) Σ_k A[t][k]·W[r][k]   — 64x64 output tiles, 16-deep k slabs, 4x4 per thread
template <typename WT>
__global__ void __launch_bounds__(256) k_gemm(const float* __restrict__ A, const WT* __restrict__ W,
                                              float* __restrict__ Y, int T, int M, int K, int add) {
  __shared__ float As[16][64 + 4];
  __shared__ float Ws[16][64 + 4];
  const int tid = threadIdx.x;
  const int tx = tid & 15, ty = tid >> 4;
  const int r0 = blockIdx.x * 64, t0 = blockIdx.y * 64;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += 16) {
    // A tile: 64 positions x 16 k ; W tile: 64 rows x 16 k  (4 elements per thread each)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int idx = tid + i * 256;
      const int rr = idx >> 4, kk = idx & 15;
      const int t = t0 + rr, r = r0 + rr;
      As[kk][rr] = (t < T) ? A[static_cast<size_t>(t) * K + k0 + kk] : 0.f;
      float wv = 0.f;
      if (r < M) {
        if constexpr (sizeof(WT) == 2) wv = bf16_to_f(reinterpret_cast<const uint16_t*>(W)[static_cast<size_t>(r) * K + k0 + kk]);
        else wv = reinterpret_cast<const float*>(W)[static_cast<size_t>(r) * K + k0 + kk];
      }
      Ws[kk][rr] = wv;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      float a[4], w[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        a[i] = As[kk][ty * 4 + i];
        w[i] = Ws[kk][tx * 4 + i];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], w[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = t0 + ty * 4 + i;
    if (t >= T) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int r = r0 + tx * 4 + j;
      if (r >= M) continue;
      float* y = Y + static_cast<size_t>(t) * M + r;
      *y = add ? (*y + acc[i][j]) : acc[i][j];
    }
  }
}

__global__ void k_swiglu(float* a, const float* b, size_t n) {
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const float x = a[i];
    a[i] = (x / (1.0f + expf(-x))) * b[i];
  }
}

// per-head RMSNorm + RoPE for q (in place) and k; K/V stored (rounded to the cache type) at
// slot pos0 + t.  One warp per (position, head among q heads then k heads).
template <typename KT, int HD>
__global__ void k_qk_rope_kv(float* QKV, int T, int pos0, Dims d, const void* qn, const void* kn,
                             const float2* rope, KT* Kc, KT* Vc, int slots) {
  constexpr int DPL = HD / 32;
  const int lane = threadIdx.x & 31;
  const int item = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int nh = d.Hq + d.Hkv;
  if (item >= T * nh) return;
  const int t = item / nh, h = item % nh;
  const int pos = pos0 + t;
  const int QD = (d.Hq + 2 * d.Hkv) * HD;
  float* row = QKV + static_cast<size_t>(t) * QD;
  float v[DPL];
#pragma unroll
  for (int j = 0; j < DPL; ++j) v[j] = row[h * HD + lane * DPL + j];
  if (d.qk_norm) {
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < DPL; ++j) s += v[j] * v[j];
    s = warp_sum(s);
    const float r = 1.0f / sqrtf(s / static_cast<float>(HD) + d.eps);
    const void* nw = h < d.Hq ? qn : kn;
#pragma unroll
    for (int j = 0; j < DPL; ++j) v[j] = (v[j] * r) * wload(nw, lane * DPL + j, d.esz);
  }
  const float2* rr = rope + static_cast<size_t>(pos) * (HD / 2);
#pragma unroll
  for (int j = 0; j < DPL; j += 2) {
    const float2 cs = rr[(lane * DPL + j) >> 1];
    const float a = v[j], b = v[j + 1];
    v[j] = a * cs.x - b * cs.y;
    v[j + 1] = a * cs.y + b * cs.x;
  }
  if (h < d.Hq) {
#pragma unroll
    for (int j = 0; j < DPL; ++j) row[h * HD + lane * DPL + j] = v[j];
  } else {
    const int g = h - d.Hq;
    KT* kd = Kc + (static_cast<size_t>(g) * slots + pos) * HD + lane * DPL;
    KT* vd = Vc + (static_cast<size_t>(g) * slots + pos) * HD + lane * DPL;
#pragma unroll
    for (int j = 0; j < DPL; ++j) {
      if constexpr (sizeof(KT) == 2) {
        kd[j] = __float2half_rn(v[j]);
        vd[j] = __float2half_rn(row[(d.Hq + d.Hkv + g) * HD + lane * DPL + j]);
      } else {
        kd[j] = v[j];
        vd[j] = row[(d.Hq + d.Hkv + g) * HD + lane * DPL + j];
      }
    }
  }
}

template <typename KT>
__device__ __forceinline__ void load_row(const KT* p, float* out, int n) {
  for (int i = 0; i < n; ++i) {
    if constexpr (sizeof(KT) == 2) out[i] = __half2float(p[i]);
    else out[i] = p[i];
  }
}

// Causal attention of position t (slot pos0+t) over slots 0..pos0+t for the rep query heads of
// KV head g.  One warp per (t, g): lane-per-slot scores, online softmax, P·V with shuffles.
template <typename KT, int HD>
__global__ void __launch_bounds__(256) k_attn_prefill(const float* QKV, int T, int pos0, Dims d, const KT* Kc,
                                                      const KT* Vc, int slots, float scale, float* O) {
  constexpr int DPL = HD / 32;
  __shared__ float qs[8][4][HD];
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int item = blockIdx.x * 8 + w;
  const int rep = d.Hq / d.Hkv;
  if (item >= T * d.Hkv) return;
  const int t = item / d.Hkv, g = item % d.Hkv;
  const int n = pos0 + t + 1;
  const int QD = (d.Hq + 2 * d.Hkv) * HD;
  for (int r = 0; r < rep; ++r)
    for (int e = lane; e < HD; e += 32) qs[w][r][e] = QKV[static_cast<size_t>(t) * QD + (g * rep + r) * HD + e];
  __syncwarp();
  float mr[4], lr[4], acc[4][DPL];
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    mr[r] = -INFINITY;
    lr[r] = 0.f;
#pragma unroll
    for (int j = 0; j < DPL; ++j) acc[r][j] = 0.f;
  }
  const KT* Kg = Kc + static_cast<size_t>(g) * slots * HD;
  const KT* Vg = Vc + static_cast<size_t>(g) * slots * HD;
  for (int b0 = 0; b0 < n; b0 += 32) {
    const int nvalid = min(32, n - b0);
    const bool valid = lane < nvalid;
    float sc[4] = {0.f, 0.f, 0.f, 0.f};
    if (valid) {
      const KT* kr = Kg + static_cast<size_t>(b0 + lane) * HD;
      for (int e0 = 0; e0 < HD; e0 += 8) {
        float kf[8];
        load_row<KT>(kr + e0, kf, 8);
#pragma unroll
        for (int tt = 0; tt < 8; ++tt)
#pragma unroll
          for (int r = 0; r < 4; ++r)
            if (r < rep) sc[r] = fmaf(qs[w][r][e0 + tt], kf[tt], sc[r]);
      }
    }
    float p[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      if (r >= rep) continue;
      const float s_ = valid ? sc[r] * scale : -INFINITY;
      const float mnew = fmaxf(mr[r], warp_max(s_));
      const float alpha = expf(mr[r] - mnew);
      p[r] = valid ? expf(s_ - mnew) : 0.f;
      lr[r] = lr[r] * alpha + warp_sum(p[r]);
#pragma unroll
      for (int j = 0; j < DPL; ++j) acc[r][j] *= alpha;
      mr[r] = mnew;
    }
    for (int jj = 0; jj < nvalid; ++jj) {
      float vv[DPL];
      load_row<KT>(Vg + static_cast<size_t>(b0 + jj) * HD + lane * DPL, vv, DPL);
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        if (r >= rep) continue;
        const float pj = __shfl_sync(0xffffffffu, p[r], jj);
#pragma unroll
        for (int j = 0; j < DPL; ++j) acc[r][j] = fmaf(pj, vv[j], acc[r][j]);
      }
    }
  }
  for (int r = 0; r < rep; ++r)
#pragma unroll
    for (int j = 0; j < DPL; ++j)
      O[static_cast<size_t>(t) * d.Hq * HD + (g * rep + r) * HD + lane * DPL + j] = acc[r][j] / lr[r];
}

// final RMSNorm of the last position and tied logits on the admissible ids
// (sem_begin..sem_end, then im_end) — one warp per output row.
__global__ void k_final(const float* x, Dims d, const void* normw, const void* E, float* hidden, float* logits) {
  extern __shared__ float hs[];
  __shared__ float sh[32];
  float s = 0.f;
  for (int e = threadIdx.x; e < d.D; e += blockDim.x) s += x[e] * x[e];
  const float tot = block_sum(s, sh);
  const float r = 1.0f / sqrtf(tot / static_cast<float>(d.D) + d.eps);
  for (int e = threadIdx.x; e < d.D; e += blockDim.x) {
    hs[e] = (x[e] * r) * wload(normw, e, d.esz);
    if (blockIdx.x == 0) hidden[e] = hs[e];
  }
  __syncthreads();
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int i = blockIdx.x * (blockDim.x >> 5) + w;
  if (i >= d.A) return;
  const int id = i < d.cbs ? d.sem_lo + i : d.im_end;
  float acc = 0.f;
  for (int e = lane; e < d.D; e += 32) acc = fmaf(wload(E, static_cast<size_t>(id) * d.D + e, d.esz), hs[e], acc);
  acc = warp_sum(acc);
  if (lane == 0) logits[i] = acc;
}

__global__ void k_state_reset(StreamState* st, int T) {
  if (threadIdx.x != 0) return;
  st->pos = T;
  st->frames_done = 0;
  st->done = 0;
  st->prefilled = 1;
  st->wlen = 0;
  st->n_out = 0;
  st->status = 0;
  st->stop_req = 0;
}

// cos/sin of pos·θ_i, θ_i = base^(-2i/hd), formed in fp64, rounded to fp32 (then bf16)
__global__ void k_rope_table(float2* tab, int npos, int hd, double base, int bf16) {
  const int half = hd / 2;
  const size_t n = static_cast<size_t>(npos) * half;
  for (size_t k = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; k < n;
       k += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const int p = static_cast<int>(k / half), i = static_cast<int>(k % half);
    const double theta = pow(base, -2.0 * static_cast<double>(i) / static_cast<double>(hd));
    const double ang = static_cast<double>(p) * theta;
    float c = static_cast<float>(cos(ang)), s = static_cast<float>(sin(ang));
    if (bf16) {
      c = round_bf16(c);
      s = round_bf16(s);
    }
    tab[k] = make_float2(c, s);
  }
}

__global__ void k_compact(const int32_t* stage, int32_t* codes, const StreamState* st, int ncb, int32_t* n_out) {
  const int n = st->n_out;
  for (int idx = threadIdx.x; idx < n * ncb; idx += blockDim.x) {
    const int cb = idx / n, f = idx % n;
    codes[idx] = stage[static_cast<size_t>(f) * ncb + cb];
    (void)cb;
  }
  if (threadIdx.x == 0) *n_out = n;
}

// tensor-core prompt projections: the rows of a chunk as bf16 hi / lo planes (rows 2t, 2t+1) of
// RMSNorm(x_t)·w, or of x_t itself when w is null
__global__ void __launch_bounds__(kBlk) k_pf_planes(const float* X, int ldx, int K, const void* w, int esz, float eps,
                                                    uint16_t* P, int ldp) {
  __shared__ float sh[32];
  const int t = blockIdx.x;
  const float* x = X + static_cast<size_t>(t) * ldx;
  float r = 1.f;
  if (w) {
    float s = 0.f;
    for (int k = threadIdx.x; k < K; k += blockDim.x) s += x[k] * x[k];
    r = 1.0f / sqrtf(block_sum(s, sh) / static_cast<float>(K) + eps);
  }
  for (int k = threadIdx.x; k < K; k += blockDim.x) {
    const float n = w ? (x[k] * r) * wload(w, k, esz) : x[k];
    const __nv_bfloat16 hi = __float2bfloat16_rn(n);
    P[static_cast<size_t>(2 * t) * ldp + k] = __bfloat16_as_ushort(hi);
    P[static_cast<size_t>(2 * t + 1) * ldp + k] = __bfloat16_as_ushort(__float2bfloat16_rn(n - __bfloat162float(hi)));
  }
}

// Y[t][m] = (add ? Y[t][m] : 0) + Σ_s part[(s*NC + t)*M + m], splits summed in order
__global__ void k_pf_reduce(const float* __restrict__ part, int splits, int NC, int M, float* Y, int ldy, int add) {
  const int t = blockIdx.y;
  for (int m = blockIdx.x * blockDim.x + threadIdx.x; m < M; m += gridDim.x * blockDim.x) {
    float a = 0.f;
    for (int s = 0; s < splits; ++s) a += __ldcg(part + (static_cast<size_t>(s) * NC + t) * M + m);
    float* y = Y + static_cast<size_t>(t) * ldy + m;
    *y = add ? *y + a : a;
  }
}

// planes of silu(Σ W1 partials)·(Σ W3 partials) (ch.02 §3.2 SwiGLU)
__global__ void k_pf_swiglu(const float* __restrict__ part, int splits, int NC, int M, uint16_t* P, int ldp) {
  const int t = blockIdx.y;
  for (int m = blockIdx.x * blockDim.x + threadIdx.x; m < M; m += gridDim.x * blockDim.x) {
    float a = 0.f, u = 0.f;
    for (int s = 0; s < splits; ++s) {
      a += __ldcg(part + (static_cast<size_t>(s) * NC + t) * M + m);
      u += __ldcg(part + (static_cast<size_t>(splits + s) * NC + t) * M + m);
    }
    const float h = (a / (1.0f + expf(-a))) * u;
    const __nv_bfloat16 hi = __float2bfloat16_rn(h);
    P[static_cast<size_t>(2 * t) * ldp + m] = __bfloat16_as_ushort(hi);
    P[static_cast<size_t>(2 * t + 1) * ldp + m] = __bfloat16_as_ushort(__float2bfloat16_rn(h - __bfloat162float(hi)));
  }
}

template <typename WT>
void gemm(const float* A, const void* W, float* Y, int T, int M, int K, int add, cudaStream_t s) {
  dim3 grid((M + 63) / 64, (T + 63) / 64);
  k_gemm<WT><<<grid, 256, 0, s>>>(A, static_cast<const WT*>(W), Y, T, M, K, add);
}

}  // namespace

size_t prefill_scratch_floats(const Dims& d, int chunk) {
  const size_t per = 2 * static_cast<size_t>(d.D) + static_cast<size_t>(d.Hq + 2 * d.Hkv) * d.hd +
                     static_cast<size_t>(d.Hq) * d.hd + 2 * static_cast<size_t>(d.F);
  return per * chunk;
}

template <typename WT, typename KT, int HD>
static int prefill_t(const PrefillArgs& a, cudaStream_t s, int* err) {
  const Dims& d = a.d;
  const int C = d.ncb + 1;
  const int QD = (d.Hq + 2 * d.Hkv) * HD;
  float* X = a.scratch;
  float* H = X + static_cast<size_t>(a.chunk) * d.D;
  float* QKV = H + static_cast<size_t>(a.chunk) * d.D;
  float* O = QKV + static_cast<size_t>(a.chunk) * QD;
  float* Ab = O + static_cast<size_t>(a.chunk) * d.Hq * HD;
  float* Bb = Ab + static_cast<size_t>(a.chunk) * d.F;
  const float scale = static_cast<float>(1.0 / sqrt(static_cast<double>(HD)));
  const bool tc = a.tc != nullptr && sizeof(WT) == 2;
  const int chunk = tc ? std::min(a.chunk, kPrefillChunkTC) : a.chunk;
  // projection y[t] = W·in[t] of the chunk: tensor cores (planes + split partials) or the fp32 tiles
  auto proj = [&](const float* in, int ldin, const void* normw, const void* W, const void* W3, float* out, int M, int K,
                  int Tc, int add) -> bool {
    if (!tc) {
      if (W3) return false;
      gemm<WT>(in, W, out, Tc, M, K, add, s);
      return true;
    }
    k_pf_planes<<<Tc, kBlk, 0, s>>>(in, ldin, K, normw, d.esz, d.eps, a.tc_planes, a.tc_ld);
    const int sp = batch_prefill_proj(a.tc, W, W3, M, K, a.tc_planes, a.tc_ld, Tc, a.tc_part, s);
    if (sp <= 0) return false;
    if (W3)
      k_pf_swiglu<<<dim3((M + 255) / 256, Tc), 256, 0, s>>>(a.tc_part, sp, Tc, M, a.tc_planes, a.tc_ld);
    else
      k_pf_reduce<<<dim3((M + 255) / 256, Tc), 256, 0, s>>>(a.tc_part, sp, Tc, M, out, M, add);
    return true;
  };
  for (int c0 = 0; c0 < a.T; c0 += chunk) {
    const int Tc = std::min(chunk, a.T - c0);
    k_embed<<<Tc, kBlk, 0, s>>>(a.tokens + static_cast<size_t>(c0) * C, Tc, d, a.E, a.CE, X, err);
    for (int l = 0; l < d.L; ++l) {
      const LayerW& w = a.layers[l];
      KT* Kc = reinterpret_cast<KT*>(static_cast<unsigned char*>(a.kc0) + l * a.kv_layer_stride);
      KT* Vc = reinterpret_cast<KT*>(static_cast<unsigned char*>(a.vc0) + l * a.kv_layer_stride);
      if (tc) {
        if (!proj(X, d.D, w.an, w.wqkv, nullptr, QKV, QD, d.D, Tc, 0)) return S2_ECUDA;
      } else {
        k_rmsnorm<<<Tc, kBlk, 0, s>>>(X, d.D, w.an, d.esz, d.eps, H);
        gemm<WT>(H, w.wqkv, QKV, Tc, QD, d.D, 0, s);
      }
      {
        const int items = Tc * (d.Hq + d.Hkv);
        k_qk_rope_kv<KT, HD><<<(items + 7) / 8, 256, 0, s>>>(QKV, Tc, c0, d, w.qn, w.kn, a.rope, Kc, Vc, a.kv_slots);
      }
      if (!(tc && sizeof(KT) == 2 && batch_prefill_attn(QKV, Tc, c0, d, Kc, Vc, a.kv_slots, scale, O, s) == 0)) {
        const int items = Tc * d.Hkv;
        k_attn_prefill<KT, HD><<<(items + 7) / 8, 256, 0, s>>>(QKV, Tc, c0, d, Kc, Vc, a.kv_slots, scale, O);
      }
      if (tc) {
        // out-projection + residual; RMSNorm + gate/up (SwiGLU planes); down-projection + residual
        if (!proj(O, d.Hq * HD, nullptr, w.wo, nullptr, X, d.D, d.Hq * HD, Tc, 1) ||
            !proj(X, d.D, w.fn, w.w1, w.w3, nullptr, d.F, d.D, Tc, 0))
          return S2_ECUDA;
        const int sp = batch_prefill_proj(a.tc, w.w2, nullptr, d.D, d.F, a.tc_planes, a.tc_ld, Tc, a.tc_part, s);
        if (sp <= 0) return S2_ECUDA;
        k_pf_reduce<<<dim3((d.D + 255) / 256, Tc), 256, 0, s>>>(a.tc_part, sp, Tc, d.D, X, d.D, 1);
      } else {
        gemm<WT>(O, w.wo, X, Tc, d.D, d.Hq * HD, 1, s);
        k_rmsnorm<<<Tc, kBlk, 0, s>>>(X, d.D, w.fn, d.esz, d.eps, H);
        gemm<WT>(H, w.w1, Ab, Tc, d.F, d.D, 0, s);
        gemm<WT>(H, w.w3, Bb, Tc, d.F, d.D, 0, s);
        k_swiglu<<<1024, 256, 0, s>>>(Ab, Bb, static_cast<size_t>(Tc) * d.F);
        gemm<WT>(Ab, w.w2, X, Tc, d.D, d.F, 1, s);
      }
    }
    if (c0 + Tc == a.T) {
      const int blocks = (d.A + 7) / 8;
      k_final<<<blocks, 256, d.D * sizeof(float), s>>>(X + static_cast<size_t>(Tc - 1) * d.D, d, a.norm, a.E,
                                                        a.hidden, a.logits);
    }
  }
  k_state_reset<<<1, 32, 0, s>>>(a.st, a.T);
  return cudaGetLastError() == cudaSuccess ? S2_OK : S2_ECUDA;
}

int run_prefill(const PrefillArgs& a, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int* err = a.err;
  const Dims& d = a.d;
  if (d.wdt == S2_BF16) {
    if (d.kvdt == S2_F16) return d.hd == 128 ? prefill_t<uint16_t, __half, 128>(a, s, err) : prefill_t<uint16_t, __half, 64>(a, s, err);
    return d.hd == 128 ? prefill_t<uint16_t, float, 128>(a, s, err) : prefill_t<uint16_t, float, 64>(a, s, err);
  }
  if (d.kvdt == S2_F16) return d.hd == 128 ? prefill_t<float, __half, 128>(a, s, err) : prefill_t<float, __half, 64>(a, s, err);
  return d.hd == 128 ? prefill_t<float, float, 128>(a, s, err) : prefill_t<float, float, 64>(a, s, err);
}

int run_head(const Dims& d, const float* x, const void* norm, const void* E, float* hidden, float* logits,
             StreamState* st, int pos, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int blocks = (d.A + 7) / 8;
  k_final<<<blocks, 256, d.D * sizeof(float), s>>>(x, d, norm, E, hidden, logits);
  k_state_reset<<<1, 32, 0, s>>>(st, pos);
  return cudaGetLastError() == cudaSuccess ? S2_OK : S2_ECUDA;
}

int build_rope_tables(float2* slow, int slots, int hd, float2* fast, int wf, int hdf, double base, int bf16,
                      void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (slots > 0) k_rope_table<<<1024, 256, 0, s>>>(slow, slots, hd, base, bf16);
  k_rope_table<<<64, 256, 0, s>>>(fast, wf, hdf, base, bf16);
  return cudaGetLastError() == cudaSuccess ? S2_OK : S2_ECUDA;
}

int compact_codes(const int32_t* stage, int32_t* codes, const StreamState* st, int n_frames, int ncb,
                  int32_t* n_out, void* stream) {
  (void)n_frames;
  k_compact<<<1, 1024, 0, static_cast<cudaStream_t>(stream)>>>(stage, codes, st, ncb, n_out);
  return cudaGetLastError() == cudaSuccess ? S2_OK : S2_ECUDA;
}

}  // namespace s2
