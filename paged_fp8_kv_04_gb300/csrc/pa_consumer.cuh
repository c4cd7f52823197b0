// pa_consumer.cuh -- the consumer warps: attention over one KV tile at a time.
//
// Fragment layout of the FP8 path (mma.sync m16n8k16, f16 in, f32 accumulate; lane
// = 4 g + t).  The reduction index of each product may be permuted freely, so it is
// chosen to make every operand load a plain 16-byte shared-memory read:
//  * QK^T: m-tile rows are the 16 query heads of one query token; n is the token.
//    For k-step kk, lane (g, t) holds k-slots {2t, 2t+1, 2t+8, 2t+9} mapped to
//    head-dim d = 32t + 4kk + {0, 1, 2, 3}, so its K operand for token g is the 4
//    bytes at d = 32t + 4kk of that token's row: one 32-byte run covers all 8 k-steps.
//  * PV: n-tile i column g is d = 16g + i, so lane (g, t) reads the 16 bytes
//    d = 16g .. 16g + 15 of the token rows 2t, 2t+1, 2t+8, 2t+9 and interleaves row
//    pairs with byte permutes into (token, token+1) pairs per d.
//  * The output accumulator o[i][e] (e = 0, 1 row g; e = 2, 3 row g + 8) holds
//    d = 32t + i (e even) and d = 32t + 16 + i (e odd).
// e4m3 codes widen to f16 exactly (the conversion instruction is exact), so the FP8
// cache enters the tensor cores unrounded; the query is rounded bf16 -> f16, exact for
// 2^-17 <= |q| <= 65504 (values above are flagged).
// The BF16 path keeps the natural d order and uses ldmatrix for its operands.
#pragma once

#include <cuda_bf16.h>

#include "pa_kernel.cuh"

namespace pa {

struct Frag {
  uint32_t qf[8][4];
  float o[16][4];
  float m[2], l[2];
  int pe[2];  // per-token V scales: row g's (pe[0]) and row g + 8's (pe[1]) o and P' are in
              // units of 2^pe (online_row_pe)
};

__device__ __forceinline__ float quad_sum(float v) {
  v += __shfl_xor_sync(~0u, v, 1);
  v += __shfl_xor_sync(~0u, v, 2);
  return v;
}

// d index of accumulator element o[i][e] for lane quad position t.
template <int KVT>
__device__ __forceinline__ int dmap(int i, int e, int t) {
  if (KVT == PA_KV_FP8_E4M3) return 32 * t + 16 * (e & 1) + i;
  return 8 * i + 2 * t + (e & 1);
}

// Bounded barrier among the 8 consumer warps (an mbarrier; named barriers cannot give up).
__device__ __forceinline__ void cons_sync(const KParams &p, const Smem &sm, uint32_t &phase) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(sm.consbar());
  if (!mbar_wait_bounded(sm.consbar(), phase)) {
    if ((threadIdx.x & 31) == 0) raise_flag(p, sm, PA_DEV_TIMEOUT);
  }
  phase ^= 1u;
}

// ----------------------------------------------------------------------------- queries

template <int KVT>
__device__ __forceinline__ void load_q(const KParams &p, uint32_t qb, int g, int t, Frag &f) {
  uint32_t bad = 0;
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const uint32_t rowb = qb + (g + 8 * half) * (kD * 2);
    if (KVT == PA_KV_FP8_E4M3) {
      uint32_t w[16];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint4 v = lds128(rowb + 64 * t + 16 * k);
        w[4 * k] = v.x;
        w[4 * k + 1] = v.y;
        w[4 * k + 2] = v.z;
        w[4 * k + 3] = v.w;
      }
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const float lo = bf16lo(w[j]), hi = bf16hi(w[j]);
        bad |= (fabsf(lo) > 65504.f) | (fabsf(hi) > 65504.f);
        f.qf[j >> 1][(j & 1) * 2 + half] = pack_f16x2(lo, hi);
      }
    } else {
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        uint32_t a0, a2;
        asm volatile("ld.shared.b32 %0, [%1];" : "=r"(a0) : "r"(rowb + 32 * kk + 4 * t));
        asm volatile("ld.shared.b32 %0, [%1];" : "=r"(a2) : "r"(rowb + 32 * kk + 16 + 4 * t));
        f.qf[kk][half] = a0;
        f.qf[kk][2 + half] = a2;
      }
    }
  }
  if (bad) atomicOr(p.status, PA_DEV_Q_RANGE);
}

__device__ __forceinline__ void reset_state(Frag &f) {
#pragma unroll
  for (int i = 0; i < 16; ++i)
#pragma unroll
    for (int e = 0; e < 4; ++e) f.o[i][e] = 0.f;
  f.m[0] = f.m[1] = -INFINITY;
  f.l[0] = f.l[1] = 0.f;
  f.pe[0] = f.pe[1] = 0;
}

// Per-token V scales fold into P per row: P'[j] = p[j] * v_scale[j] * 2^pe, with one power
// of two per row (and lane quad), so that P' never overflows the f16 operand however far
// apart the tokens' magnitudes are (per-token scales of 2^-20 .. 2^20 in one sequence
// included).  The row's o is accumulated in the same units, and the power of two rides in
// the exponent of p.  A chunk keeps the rows' powers of two while every weight * 2^pe lies
// in [2^-3, 2^12): no product reaches 2^12, and the row's p = 1 token, wherever it is,
// contributes at least 2^-3, so what f16's subnormals can lose on the smallest products
// stays below 2^-22 of the row's sum per token.  Otherwise pe is placed anew: from the
// chunk's V-scale exponent range and the row's largest p' (online_row_fit), known before
// the exponentials, so that the largest products keep f16's 11 bits; a chunk whose scales
// spread wider than 2^15 (or that holds masked tokens) takes an exact placement on its P'
// (refold_row).  The reference is the largest product, not the largest scale, so a token
// with p = 1 and a small scale is not flushed by a neighbour with a large scale and p ~ 0.
// pe stays within [-60, 60], which covers V scales of 2^-60 .. 2^64.
constexpr int kPeMin = -60, kPeMax = 60;
constexpr int kScalarPe = 8;  // the fixed power of two of P in scalar-scale mode

// The online softmax step of one row with p' = 2^(s - m + pe) = p * 2^pe in s on return
// (l still sums p); returns the factor the row's accumulators must be rescaled by (1 when
// the maximum did not grow).
template <int N>
__device__ __forceinline__ float online_row_pe(float (&s)[N], float &m, float &l, int pe) {
  float mx = s[0];
#pragma unroll
  for (int k = 1; k < N; ++k) mx = fmaxf(mx, s[k]);
  mx = fmaxf(mx, __shfl_xor_sync(~0u, mx, 1));
  mx = fmaxf(mx, __shfl_xor_sync(~0u, mx, 2));
  float alpha = 1.f;
  if (mx > m) {
    alpha = fast_exp2(m - mx);
    m = mx;
    l *= alpha;
  }
  const float ref = ((m == -INFINITY) ? 0.f : m) - (float)pe;
#pragma unroll
  for (int k = 0; k < N; ++k) s[k] = fast_exp2(s[k] - ref);
  float sum = 0.f;
#pragma unroll
  for (int k = 0; k < N; k += 4) sum += (s[k] + s[k + 1]) + (s[k + 2] + s[k + 3]);
  l += sum * __uint_as_float((uint32_t)(127 - pe) << 23);
  return alpha;
}

// floor(log2 x) of a positive normal float, from its exponent field; -1000 for 0.
__device__ __forceinline__ int ilog2f(float x) {
  return x > 0.f ? (int)((__float_as_uint(x) >> 23) & 0xFFu) - 127 : -1000;
}

// floor(log2) of the smallest and the largest of the chunk's V weights.  Every lane quad
// holds all of the chunk's tokens, so a reduction over the whole warp (one redux per
// bound) gives the chunk's range, the same in every lane.
template <int N>
__device__ __forceinline__ void weight_exponents(const float (&w)[N], int &el, int &eh) {
  float a[N / 2], b[N / 2];
#pragma unroll
  for (int k = 0; k < N / 2; ++k) {
    a[k] = fminf(w[2 * k], w[2 * k + 1]);
    b[k] = fmaxf(w[2 * k], w[2 * k + 1]);
  }
#pragma unroll
  for (int n = N / 4; n >= 1; n >>= 1) {  // a tree: log2 N dependent steps
#pragma unroll
    for (int k = 0; k < n; ++k) {
      a[k] = fminf(a[k], a[k + n]);
      b[k] = fmaxf(b[k], b[k + n]);
    }
  }
  el = __reduce_min_sync(~0u, ilog2f(a[0]));
  eh = __reduce_max_sync(~0u, ilog2f(b[0]));
}

// online_row_pe for a chunk whose V weights lie in [2^el, 2^(eh + 1)) with eh - el <= 15:
// the row's largest P' then lies in [2^(top + el), 2^(top + eh + 1)), top the log2 of its
// largest p'.  When that interval leaves the window [2^-6, 2^12), pe moves (and the
// returned factor rescales o) so that its upper end lands in (2^(T - 1), 2^T], T = (7 +
// eh - el) / 2, the middle of the room the window leaves; its lower end then stays above
// 2^-6.  No test of P' itself, and no branch between the softmax and PV.
template <int N>
__device__ __forceinline__ float online_row_fit(float (&s)[N], float &m, float &l, int &pe,
                                                int eh, int el) {
  float mx = s[0];
#pragma unroll
  for (int k = 1; k < N; ++k) mx = fmaxf(mx, s[k]);
  mx = fmaxf(mx, __shfl_xor_sync(~0u, mx, 1));
  mx = fmaxf(mx, __shfl_xor_sync(~0u, mx, 2));
  float alpha = 1.f;
  if (mx > m) {
    alpha = fast_exp2(m - mx);
    m = mx;
    l *= alpha;
  }
  if (mx != -INFINITY) {
    const float top = mx - m + (float)pe;
    const float hb = top + (float)(eh + 1), lb = top + (float)el;
    if (hb > 12.f || lb < -6.f) {
      const int T = (7 + eh - el) >> 1;
      const int ne = min(max(pe + T - (int)ceilf(hb), kPeMin), kPeMax);
      alpha *= __uint_as_float((uint32_t)(ne - pe + 127) << 23);
      pe = ne;
    }
  }
  const float ref = ((m == -INFINITY) ? 0.f : m) - (float)pe;
#pragma unroll
  for (int k = 0; k < N; ++k) s[k] = fast_exp2(s[k] - ref);
  float sum = 0.f;
#pragma unroll
  for (int k = 0; k < N; k += 4) sum += (s[k] + s[k + 1]) + (s[k + 2] + s[k + 3]);
  l += sum * __uint_as_float((uint32_t)(127 - pe) << 23);
  return alpha;
}

// The row's P' (in s, fp32) checked against the window [2^-6, 2^12): outside it, a new pe
// from the fp32 maximum that puts it in [2^6, 2^7) (0 keeps it).  Returns the factor P' and
// the row's o are rescaled by.
template <int N>
__device__ __forceinline__ float refold_row(float (&s)[N], int &pe) {
  float wmax = 0.f;
#pragma unroll
  for (int k = 0; k < N; ++k) wmax = fmaxf(wmax, s[k]);
  wmax = fmaxf(wmax, __shfl_xor_sync(~0u, wmax, 1));
  wmax = fmaxf(wmax, __shfl_xor_sync(~0u, wmax, 2));
  float rs = 1.f;
  if (wmax > 0.f) {
    const int ev = (int)((__float_as_uint(wmax) >> 23) & 0xFFu) - 127;  // floor(log2 wmax)
    if (ev < -6 || ev > 11) {
      const int ne = min(min(max(pe + 6 - ev, kPeMin), kPeMax), pe + 64);
      const int d = ne - pe;
      rs = d < -126 ? 0.f : __uint_as_float((uint32_t)(d + 127) << 23);
      pe = ne;
#pragma unroll
      for (int k = 0; k < N; ++k) s[k] *= rs;
    }
  }
  return rs;
}

// o back to plain units (2^-pe per row, exact) before it leaves the warp.
__device__ __forceinline__ void unfold_rows(Frag &f) {
#pragma unroll
  for (int hf = 0; hf < 2; ++hf) {
    if (f.pe[hf] == 0) continue;
    const float u = __uint_as_float((uint32_t)(127 - f.pe[hf]) << 23);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      f.o[i][2 * hf] *= u;
      f.o[i][2 * hf + 1] *= u;
    }
    f.pe[hf] = 0;
  }
}

// ------------------------------------------------------------------------ online softmax

// The online softmax step of one row.  s holds the log2-domain scores of this lane's
// columns of the row (tokens 8j + 2t + e of the chunk's n-tiles j, column 2j + e); on
// return it holds p = 2^(s - m) with m the row's running maximum, l is updated, and the
// row's accumulators (o[.][half], o[.][half + 1]) are rescaled in the same branch when the
// maximum grew.  For paths whose P needs no further fold.
template <int N>
__device__ __forceinline__ void online_row_rescale(float (&s)[N], float &m, float &l,
                                                   float (&o)[16][4], int half) {
  float mx = s[0];
#pragma unroll
  for (int k = 1; k < N; ++k) mx = fmaxf(mx, s[k]);
  mx = fmaxf(mx, __shfl_xor_sync(~0u, mx, 1));
  mx = fmaxf(mx, __shfl_xor_sync(~0u, mx, 2));
  if (mx > m) {
    const float alpha = fast_exp2(m - mx);
    m = mx;
    l *= alpha;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      o[i][half] *= alpha;
      o[i][half + 1] *= alpha;
    }
  }
  const float ref = (m == -INFINITY) ? 0.f : m;
#pragma unroll
  for (int k = 0; k < N; ++k) s[k] = fast_exp2(s[k] - ref);
  float sum = 0.f;
#pragma unroll
  for (int k = 0; k < N; k += 4) sum += (s[k] + s[k + 1]) + (s[k + 2] + s[k + 3]);
  l += sum;
}

// Rescales the accumulators of row g by a0 and of row g + 8 by a1.
__device__ __forceinline__ void rescale_rows(float (&o)[16][4], float a0, float a1) {
  if (a0 != 1.f) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      o[i][0] *= a0;
      o[i][1] *= a0;
    }
  }
  if (a1 != 1.f) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      o[i][2] *= a1;
      o[i][3] *= a1;
    }
  }
}

// Masks the columns whose position is not below the row's cutoff.  pos0[h] is the
// position of token 2t of the chunk's 16-token half h, or < 0 for an empty page slot.
template <int N>
__device__ __forceinline__ void mask_scores(float (&s0)[N], float (&s1)[N],
                                            const int (&pos0)[N / 4], int cut) {
#pragma unroll
  for (int k = 0; k < N; ++k) {
    const int j = k >> 1, hf = j >> 1;
    const int pos = pos0[hf] + 8 * (j & 1) + (k & 1);
    if (pos0[hf] < 0 || pos >= cut) {
      s0[k] = -INFINITY;
      s1[k] = -INFINITY;
    }
  }
}

// The per-token V scales of the columns mask_scores masks, set to 0: an empty page slot's
// scale in shared memory is whatever an earlier tile or kernel left there, and a masked
// column's probability 0 times a NaN scale would still be NaN.
template <int N>
__device__ __forceinline__ void mask_weights(float (&w)[N], const int (&pos0)[N / 4], int cut) {
#pragma unroll
  for (int k = 0; k < N; ++k) {
    const int j = k >> 1, hf = j >> 1;
    const int pos = pos0[hf] + 8 * (j & 1) + (k & 1);
    if (pos0[hf] < 0 || pos >= cut) w[k] = 0.f;
  }
}

// P fragments of the chunk's PV k-steps from P' of rows g (s0) and g + 8 (s1).
template <int N>
__device__ __forceinline__ void pack_p(const float (&s0)[N], const float (&s1)[N], bool bf16,
                                       uint32_t (&pa)[N / 4][4]) {
#pragma unroll
  for (int ks = 0; ks < N / 4; ++ks) {
    const int c = 4 * ks;
    if (bf16) {
      pa[ks][0] = pack_bf16x2(s0[c], s0[c + 1]);
      pa[ks][1] = pack_bf16x2(s1[c], s1[c + 1]);
      pa[ks][2] = pack_bf16x2(s0[c + 2], s0[c + 3]);
      pa[ks][3] = pack_bf16x2(s1[c + 2], s1[c + 3]);
    } else {
      pa[ks][0] = pack_f16x2(s0[c], s0[c + 1]);
      pa[ks][1] = pack_f16x2(s1[c], s1[c + 1]);
      pa[ks][2] = pack_f16x2(s0[c + 2], s0[c + 3]);
      pa[ks][3] = pack_f16x2(s1[c + 2], s1[c + 3]);
    }
  }
}

// ---------------------------------------------------------------- 32 or 64-token chunks

// FP8 tile: K at st, V at st + 16384 (each [128 tokens][128 B], 128-byte swizzle),
// K scales at st + 32768, V scales at st + 33280 (fp32 per token).  Tokens tb ..
// tb + 8 NJ - 1: NJ QK n-tiles of 8 tokens (NJ independent accumulator chains) and NJ / 2
// PV k-steps of 16 tokens.
template <int SM, int NJ>
__device__ __forceinline__ void chunk_fp8(const KParams &p, uint32_t st, int tb, bool masked,
                                          const int (&pos0)[NJ / 2], int cut, int Lctx, int g,
                                          int t, Frag &f) {
  constexpr int NC = 2 * NJ, NKS = NJ / 2;
  const uint32_t Kb = st, Vb = st + 16384;
  const uint32_t sw0 = ((2 * t) ^ g) << 4, sw1 = ((2 * t + 1) ^ g) << 4;
  uint32_t w[NJ][8];
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    const uint32_t rb = Kb + (tb + 8 * j + g) * 128;
    const uint4 x = lds128(rb + sw0), y = lds128(rb + sw1);
    w[j][0] = x.x; w[j][1] = x.y; w[j][2] = x.z; w[j][3] = x.w;
    w[j][4] = y.x; w[j][5] = y.y; w[j][6] = y.z; w[j][7] = y.w;
  }
  float acc[NJ][4];
#pragma unroll
  for (int j = 0; j < NJ; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      uint32_t b0, b1;
      e4m3x4_to_f16x2x2(w[j][kk], b0, b1);
      mma_f16(acc[j], f.qf[kk], b0, b1);
    }
  }
  float c[NC], vw[NC];
  if (SM == PA_SCALE_PER_TOKEN) {
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      const float2 x = lds64f(st + 32768 + (tb + 8 * j + 2 * t) * 4);
      const float2 y = lds64f(st + 33280 + (tb + 8 * j + 2 * t) * 4);
      c[2 * j] = x.x * p.kfold;
      c[2 * j + 1] = x.y * p.kfold;
      vw[2 * j] = y.x;
      vw[2 * j + 1] = y.y;
    }
  } else {
#pragma unroll
    for (int k = 0; k < NC; ++k) {
      c[k] = p.kfold;
      vw[k] = 1.f;
    }
  }
  float s0[NC], s1[NC];
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    s0[2 * j] = acc[j][0] * c[2 * j];
    s0[2 * j + 1] = acc[j][1] * c[2 * j + 1];
    s1[2 * j] = acc[j][2] * c[2 * j];
    s1[2 * j + 1] = acc[j][3] * c[2 * j + 1];
  }
  if (masked) {
    mask_scores<NC>(s0, s1, pos0, cut);
    if (SM == PA_SCALE_PER_TOKEN) mask_weights<NC>(vw, pos0, cut);
  }
  uint32_t pa[NKS][4];
  float a0, a1;
  if (SM == PA_SCALE_PER_TOKEN) {
    // The rows' powers of two stand while every weight of the chunk keeps its products
    // below 2^12 and its p = 1 product at or above 2^-3 (a min / max over the lane's
    // weights and one vote): no search, nothing between the softmax and PV.
    float vmx = vw[0], vmn = vw[0];
#pragma unroll
    for (int k = 1; k < NC; ++k) {
      vmx = fmaxf(vmx, vw[k]);
      vmn = fminf(vmn, vw[k]);
    }
    const float u0 = __uint_as_float((uint32_t)(f.pe[0] + 127) << 23);
    const float u1 = __uint_as_float((uint32_t)(f.pe[1] + 127) << 23);
    const bool stands = !masked && vmx * u0 < 4096.f && vmx * u1 < 4096.f && vmn * u0 >= 0.125f &&
                        vmn * u1 >= 0.125f;
    if (__all_sync(~0u, stands)) {
      a0 = online_row_pe<NC>(s0, f.m[0], f.l[0], f.pe[0]);
      a1 = online_row_pe<NC>(s1, f.m[1], f.l[1], f.pe[1]);
#pragma unroll
      for (int k = 0; k < NC; ++k) {
        s0[k] *= vw[k];
        s1[k] *= vw[k];
      }
    } else {
      int el, eh;
      weight_exponents<NC>(vw, el, eh);
      if (eh - el <= 15) {  // the same for the whole warp
        a0 = online_row_fit<NC>(s0, f.m[0], f.l[0], f.pe[0], eh, el);
        a1 = online_row_fit<NC>(s1, f.m[1], f.l[1], f.pe[1], eh, el);
#pragma unroll
        for (int k = 0; k < NC; ++k) {
          s0[k] *= vw[k];
          s1[k] *= vw[k];
        }
      } else {
        // scales spread wider (or masked tokens, whose weight is 0): each row's window is
        // settled on its fp32 P'
        a0 = online_row_pe<NC>(s0, f.m[0], f.l[0], f.pe[0]);
        a1 = online_row_pe<NC>(s1, f.m[1], f.l[1], f.pe[1]);
#pragma unroll
        for (int k = 0; k < NC; ++k) {
          s0[k] *= vw[k];
          s1[k] *= vw[k];
        }
        a0 *= refold_row<NC>(s0, f.pe[0]);
        a1 *= refold_row<NC>(s1, f.pe[1]);
      }
    }
  } else {
    // one scale for the whole cache: P' = p * 2^8 (p <= 1) keeps p down to 2^-22 out of
    // f16's subnormals; the host folds 2^-8 into the V scale applied at the end
    a0 = online_row_pe<NC>(s0, f.m[0], f.l[0], kScalarPe);
    a1 = online_row_pe<NC>(s1, f.m[1], f.l[1], kScalarPe);
  }
  pack_p<NC>(s0, s1, false, pa);
  rescale_rows(f.o, a0, a1);
#pragma unroll
  for (int ks = 0; ks < NKS; ++ks) {
    const int rv = tb + 16 * ks + 2 * t;
    const uint32_t sv0 = (g ^ (2 * t)) << 4, sv1 = (g ^ (2 * t + 1)) << 4;
    uint4 va = lds128(Vb + rv * 128 + sv0), vb = lds128(Vb + (rv + 1) * 128 + sv1);
    uint4 vc = lds128(Vb + (rv + 8) * 128 + sv0), vd = lds128(Vb + (rv + 9) * 128 + sv1);
    if (masked) {
      // Slots past the context or of an empty page may hold any bytes, NaN codes
      // included, and 0 * NaN = NaN: their V rows enter the product as zeros.
      const uint4 z = make_uint4(0u, 0u, 0u, 0u);
      const int pk = pos0[ks];
      if (pk < 0 || pk >= Lctx) va = z;
      if (pk < 0 || pk + 1 >= Lctx) vb = z;
      if (pk < 0 || pk + 8 >= Lctx) vc = z;
      if (pk < 0 || pk + 9 >= Lctx) vd = z;
    }
    const uint32_t A[4] = {va.x, va.y, va.z, va.w}, Bw[4] = {vb.x, vb.y, vb.z, vb.w};
    const uint32_t C[4] = {vc.x, vc.y, vc.z, vc.w}, Dw[4] = {vd.x, vd.y, vd.z, vd.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint32_t x0, x1, y0, y1;
      e4m3x4_to_f16x2x2(prmt(A[q], Bw[q], 0x5140), x0, x1);
      e4m3x4_to_f16x2x2(prmt(C[q], Dw[q], 0x5140), y0, y1);
      mma_f16(f.o[4 * q], pa[ks], x0, y0);
      mma_f16(f.o[4 * q + 1], pa[ks], x1, y1);
      e4m3x4_to_f16x2x2(prmt(A[q], Bw[q], 0x7362), x0, x1);
      e4m3x4_to_f16x2x2(prmt(C[q], Dw[q], 0x7362), y0, y1);
      mma_f16(f.o[4 * q + 2], pa[ks], x0, y0);
      mma_f16(f.o[4 * q + 3], pa[ks], x1, y1);
    }
  }
}

// BF16 tile: K halves (d 0-63, 64-127) at st and st + 16384, V halves at st + 32768 and
// st + 49152, each [128 tokens][128 B] with 128-byte swizzle.  Tokens tb..tb+31.
__device__ __forceinline__ void chunk_bf16(const KParams &p, uint32_t st, int tb, bool masked,
                                           const int (&pos0)[2], int cut, const int32_t *page_pos,
                                           int Lctx, uint32_t zline, int g, int t, int lane,
                                           Frag &f) {
  const int mat = lane >> 3, rr = lane & 7;
  float acc[4][4];
#pragma unroll
  for (int j = 0; j < 4; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const int c16 = 2 * kk + (mat & 1);
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int row = tb + 8 * (2 * q + (mat >> 1)) + rr;
      const uint32_t addr = st + (c16 >> 3) * 16384 + row * 128 + (((c16 & 7) ^ rr) << 4);
      uint32_t r0, r1, r2, r3;
      ldsm_x4(addr, r0, r1, r2, r3);
      mma_bf16(acc[2 * q], f.qf[kk], r0, r1);
      mma_bf16(acc[2 * q + 1], f.qf[kk], r2, r3);
    }
  }
  const float k = p.kfold;
  float s0[8], s1[8];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    s0[2 * j] = acc[j][0] * k;
    s0[2 * j + 1] = acc[j][1] * k;
    s1[2 * j] = acc[j][2] * k;
    s1[2 * j + 1] = acc[j][3] * k;
  }
  if (masked) mask_scores<8>(s0, s1, pos0, cut);
  online_row_rescale<8>(s0, f.m[0], f.l[0], f.o, 0);
  online_row_rescale<8>(s1, f.m[1], f.l[1], f.o, 2);
  uint32_t pa[2][4];
  pack_p<8>(s0, s1, true, pa);
#pragma unroll
  for (int ks = 0; ks < 2; ++ks) {
    const int tok = tb + 16 * ks + 8 * (mat & 1) + rr;
    bool dead = false;  // a slot past the context or of an empty page: read a zero line
    if (masked) {
      const int pp = page_pos[tok >> p.ps_shift];
      dead = pp < 0 || pp + (tok & (p.ps - 1)) >= Lctx;
    }
#pragma unroll
    for (int j = 0; j < 16; j += 2) {
      const int c16 = j + (mat >> 1);
      const uint32_t addr =
          dead ? zline : st + 32768 + (c16 >> 3) * 16384 + tok * 128 + (((c16 & 7) ^ rr) << 4);
      uint32_t r0, r1, r2, r3;
      ldsm_x4_t(addr, r0, r1, r2, r3);
      mma_bf16(f.o[j], pa[ks], r0, r1);
      mma_bf16(f.o[j + 1], pa[ks], r2, r3);
    }
  }
}

// ------------------------------------------------------------------------ state exchange

// Exchange-buffer slot k: accumulators as [16][32 lanes][4] floats at k * 8 KB; the lanes'
// (m0, m1, l0, l1) in a 512-byte block per slot after all slots' accumulators.
__device__ __forceinline__ void put_state(const Smem &sm, int k, const Frag &f, int lane) {
  const uint32_t ob = sm.merge() + k * 8192, mb = sm.merge_ml_at(k);
#pragma unroll
  for (int i = 0; i < 16; ++i)
    sts128(ob + (i * 32 + lane) * 16,
           make_uint4(__float_as_uint(f.o[i][0]), __float_as_uint(f.o[i][1]),
                      __float_as_uint(f.o[i][2]), __float_as_uint(f.o[i][3])));
  const float v[4] = {f.m[0], f.m[1], f.l[0], f.l[1]};
#pragma unroll
  for (int j = 0; j < 4; ++j)
    asm volatile("st.shared.f32 [%0], %1;" ::"r"(mb + (j * 32 + lane) * 4), "f"(v[j]));
}

__device__ __forceinline__ void merge_state(const Smem &sm, int k, Frag &f, int lane) {
  const uint32_t ob = sm.merge() + k * 8192, mb = sm.merge_ml_at(k);
  float v[4];
#pragma unroll
  for (int j = 0; j < 4; ++j)
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v[j]) : "r"(mb + (j * 32 + lane) * 4));
  float fa[2], fb[2];
#pragma unroll
  for (int hf = 0; hf < 2; ++hf) {
    const float mn = fmaxf(f.m[hf], v[hf]);
    if (mn == -INFINITY) {
      fa[hf] = 1.f;
      fb[hf] = 0.f;
    } else {
      fa[hf] = fast_exp2(f.m[hf] - mn);
      fb[hf] = fast_exp2(v[hf] - mn);
    }
    f.m[hf] = mn;
    f.l[hf] = f.l[hf] * fa[hf] + v[2 + hf] * fb[hf];
  }
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const uint4 x = lds128(ob + (i * 32 + lane) * 16);
    f.o[i][0] = f.o[i][0] * fa[0] + __uint_as_float(x.x) * fb[0];
    f.o[i][1] = f.o[i][1] * fa[0] + __uint_as_float(x.y) * fb[0];
    f.o[i][2] = f.o[i][2] * fa[1] + __uint_as_float(x.z) * fb[1];
    f.o[i][3] = f.o[i][3] * fa[1] + __uint_as_float(x.w) * fb[1];
  }
}

// ------------------------------------------------------------------------------ outputs

__device__ __forceinline__ void store_out(const KParams &p, int64_t elem, const float *v, int n) {
  // n contiguous values starting at element index elem (n a multiple of 4; elem 4-aligned)
  if (p.out_f32) {
    float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(p.out) + elem);
    for (int k = 0; k < n / 4; ++k) dst[k] = make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
  } else {
    uint2 *dst = reinterpret_cast<uint2 *>(static_cast<uint16_t *>(p.out) + elem);
    for (int k = 0; k < n / 4; ++k)
      dst[k] = make_uint2(pack_bf16x2(v[4 * k], v[4 * k + 1]), pack_bf16x2(v[4 * k + 2], v[4 * k + 3]));
  }
}

// Final (normalised) rows of one m-tile straight from the fragments.
template <int KVT>
__device__ __forceinline__ void write_final(const KParams &p, const Frag &f, int row, int head0,
                                            int g, int t) {
  const int Hq = p.Hkv * kG;
#pragma unroll
  for (int hf = 0; hf < 2; ++hf) {
    const float lq = quad_sum(f.l[hf]);
    const float sc = lq > 0.f ? p.vpost / lq : 0.f;
    const int head = head0 + g + 8 * hf;
    const int64_t rowe = ((int64_t)row * Hq + head) * kD;
    float v[32];
    if (KVT == PA_KV_FP8_E4M3) {
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        v[i] = f.o[i][2 * hf] * sc;
        v[16 + i] = f.o[i][2 * hf + 1] * sc;
      }
      store_out(p, rowe + 32 * t, v, 32);
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float a = f.o[i][2 * hf] * sc, b = f.o[i][2 * hf + 1] * sc;
        const int64_t e = rowe + 8 * i + 2 * t;
        if (p.out_f32)
          *reinterpret_cast<float2 *>(static_cast<float *>(p.out) + e) = make_float2(a, b);
        else
          *reinterpret_cast<uint32_t *>(static_cast<uint16_t *>(p.out) + e) = pack_bf16x2(a, b);
      }
    }
    if (t == 0 && p.lse != nullptr)
      p.lse[(int64_t)row * Hq + head] = lq > 0.f ? (f.m[hf] + log2f(lq)) * kLn2 : -INFINITY;
  }
}

// Split-K partial of one m-tile: m, l per row, and the unnormalised accumulators in
// fragment order ([m-tile][i][lane][4] float4s: one coalesced 512-byte store per i).
__device__ __forceinline__ void write_partial(const KParams &p, const Frag &f, int slot,
                                              int mtile, int g, int t, int lane) {
  float4 *dst = reinterpret_cast<float4 *>(p.part_o) +
                ((int64_t)slot * (p.mmax / kG) + mtile) * (16 * 32) + lane;
#pragma unroll
  for (int i = 0; i < 16; ++i)
    __stcg(dst + i * 32, make_float4(f.o[i][0], f.o[i][1], f.o[i][2], f.o[i][3]));
  // (m_g, m_g+8, l_g, l_g+8) of the row pair of lane group g: one float4 per pair.
  const float lq0 = quad_sum(f.l[0]), lq1 = quad_sum(f.l[1]);
  if (t == 0)
    __stcg(reinterpret_cast<float4 *>(p.part_ml) + ((int64_t)slot * (p.mmax / kG) + mtile) * 8 + g,
           make_float4(f.m[0], f.m[1], lq0, lq1));
}

// Stores one unit of a merged fragment: rows g and g + 8 of query token `tok`, the two
// head-dim columns of accumulator index i for lane (g, t).
template <int KVT>
__device__ __forceinline__ void store_unit(const KParams &p, int tok, int head0, int i, int g,
                                           int t, float4 v, float s0, float s1) {
  const int Hq = p.Hkv * kG;
  const int d0 = dmap<KVT>(i, 0, t), d1 = dmap<KVT>(i, 1, t);
  const int64_t e0 = ((int64_t)tok * Hq + head0 + g) * kD, e1 = e0 + 8 * kD;
  if (p.out_f32) {
    float *o = static_cast<float *>(p.out);
    o[e0 + d0] = v.x * s0;
    o[e0 + d1] = v.y * s0;
    o[e1 + d0] = v.z * s1;
    o[e1 + d1] = v.w * s1;
  } else {
    __nv_bfloat16 *o = static_cast<__nv_bfloat16 *>(p.out);
    o[e0 + d0] = __float2bfloat16_rn(v.x * s0);
    o[e0 + d1] = __float2bfloat16_rn(v.y * s0);
    o[e1 + d0] = __float2bfloat16_rn(v.z * s1);
    o[e1 + d1] = __float2bfloat16_rn(v.w * s1);
  }
}

// The last CTA to finish a split sequence merges every partial (log-sum-exp merge).
// Lane-thread u handles fragment units u and u + 256 of an m-tile, which belong to the
// same two rows, so one batch of independent loads brings the maxima, sums and
// accumulators of up to kMergeBatch partials (12 FP8, 8 BF16, which has less register
// room): one memory round trip per batch.
template <int KVT>
__device__ void merge_partials(const KParams &p, int h, int row0, int qlen, int c_first, int n,
                               int ctid) {
  constexpr int kMergeBatch = KVT == PA_KV_FP8_E4M3 ? 12 : 8;
  const int units = qlen * kG * 32;
  const float4 *src = reinterpret_cast<const float4 *>(p.part_o);
  const int64_t slot_f4 = (int64_t)(p.mmax / kG) * 512;  // float4s per partial slot
  for (int ub = (ctid & 255); ub < units; ub += 512) {
    const int u1 = ub + 256;  // same m-tile, same lane, accumulator index + 8
    const int mt = ub >> 9, ln = ub & 31, gg = ln >> 2, tt = ln & 3;
    float M0 = -INFINITY, M1 = -INFINITY, L0 = 0.f, L1 = 0.f;
    float4 a0 = make_float4(0.f, 0.f, 0.f, 0.f), a1 = a0;
    for (int k0 = 0; k0 < n; k0 += kMergeBatch) {
      float m0[kMergeBatch], m1[kMergeBatch], l0[kMergeBatch], l1[kMergeBatch];
      float4 v0[kMergeBatch], v1[kMergeBatch];
#pragma unroll
      for (int j = 0; j < kMergeBatch; ++j) {
        if (k0 + j < n) {
          const int64_t sl = slot_of(c_first + k0 + j, c_first);
          const float4 ml = __ldcg(reinterpret_cast<const float4 *>(p.part_ml) +
                                   (sl * (p.mmax / kG) + mt) * 8 + gg);
          m0[j] = ml.x;
          m1[j] = ml.y;
          l0[j] = ml.z;
          l1[j] = ml.w;
          v0[j] = __ldcg(src + sl * slot_f4 + ub);
          v1[j] = __ldcg(src + sl * slot_f4 + u1);
        } else {
          m0[j] = m1[j] = -INFINITY;
          l0[j] = l1[j] = 0.f;
          v0[j] = v1[j] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
      float n0 = M0, n1 = M1;
#pragma unroll
      for (int j = 0; j < kMergeBatch; ++j) {
        n0 = fmaxf(n0, m0[j]);
        n1 = fmaxf(n1, m1[j]);
      }
      const float c0 = n0 == -INFINITY ? 0.f : fast_exp2(M0 - n0);
      const float c1 = n1 == -INFINITY ? 0.f : fast_exp2(M1 - n1);
      a0.x *= c0; a0.y *= c0; a0.z *= c1; a0.w *= c1;
      a1.x *= c0; a1.y *= c0; a1.z *= c1; a1.w *= c1;
      L0 *= c0;
      L1 *= c1;
#pragma unroll
      for (int j = 0; j < kMergeBatch; ++j) {
        const float w0 = n0 == -INFINITY ? 0.f : fast_exp2(m0[j] - n0);
        const float w1 = n1 == -INFINITY ? 0.f : fast_exp2(m1[j] - n1);
        a0.x += w0 * v0[j].x; a0.y += w0 * v0[j].y; a0.z += w1 * v0[j].z; a0.w += w1 * v0[j].w;
        a1.x += w0 * v1[j].x; a1.y += w0 * v1[j].y; a1.z += w1 * v1[j].z; a1.w += w1 * v1[j].w;
        L0 += w0 * l0[j];
        L1 += w1 * l1[j];
      }
      M0 = n0;
      M1 = n1;
    }
    const float s0 = L0 > 0.f ? p.vpost / L0 : 0.f, s1 = L1 > 0.f ? p.vpost / L1 : 0.f;
    const int i0 = (ub >> 5) & 15;
    store_unit<KVT>(p, row0 + mt, h * kG, i0, gg, tt, a0, s0, s1);
    store_unit<KVT>(p, row0 + mt, h * kG, i0 + 8, gg, tt, a1, s0, s1);
    if (i0 == 0 && tt == 0 && p.lse != nullptr) {
      float *lp = p.lse + (int64_t)(row0 + mt) * (p.Hkv * kG) + h * kG + gg;
      lp[0] = L0 > 0.f ? (M0 + log2f(L0)) * kLn2 : -INFINITY;
      lp[8] = L1 > 0.f ? (M1 + log2f(L1)) * kLn2 : -INFINITY;
    }
  }
}

// ------------------------------------------------------- merges at the end of a sequence

// An exchange slot in stage memory (at the CTA's last sequence end, when no tile is in
// flight): the warp's accumulators as [16][32 lanes][4] floats (fragment order), then per
// lane (m_g, m_g+8, L_g, L_g+8) with L the row's sum over the lane quad.
constexpr int kSlotBytes = 8192 + 512;
constexpr int kMaxSlots = 8;

__device__ __forceinline__ void put_slot(uint32_t base, const Frag &f, int lane) {
#pragma unroll
  for (int i = 0; i < 16; ++i)
    sts128(base + (i * 32 + lane) * 16,
           make_uint4(__float_as_uint(f.o[i][0]), __float_as_uint(f.o[i][1]),
                      __float_as_uint(f.o[i][2]), __float_as_uint(f.o[i][3])));
  const float l0 = quad_sum(f.l[0]), l1 = quad_sum(f.l[1]);
  sts128(base + 8192 + lane * 16, make_uint4(__float_as_uint(f.m[0]), __float_as_uint(f.m[1]),
                                             __float_as_uint(l0), __float_as_uint(l1)));
}

// Two log-sum-exp states of the same two rows, (M, L, a) += (m, l, x) (m in log2 units).
__device__ __forceinline__ void lse_combine(float &M0, float &M1, float &L0, float &L1, float4 &a,
                                            float m0, float m1, float l0, float l1, float4 x) {
  const float n0 = fmaxf(M0, m0), n1 = fmaxf(M1, m1);
  const float c0 = n0 == -INFINITY ? 0.f : fast_exp2(M0 - n0);
  const float c1 = n1 == -INFINITY ? 0.f : fast_exp2(M1 - n1);
  const float w0 = n0 == -INFINITY ? 0.f : fast_exp2(m0 - n0);
  const float w1 = n1 == -INFINITY ? 0.f : fast_exp2(m1 - n1);
  a.x = a.x * c0 + x.x * w0;
  a.y = a.y * c0 + x.y * w0;
  a.z = a.z * c1 + x.z * w1;
  a.w = a.w * c1 + x.w * w1;
  L0 = L0 * c0 + l0 * w0;
  L1 = L1 * c1 + l1 * w1;
  M0 = n0;
  M1 = n1;
}

// The CTA's last sequence end, all consumer threads at once: the nsl token slices of each
// of the mt m-tiles (slot s * mt + mtile at base) merged element by element.  whole: the
// normalised output rows (and lse) of the sequence; otherwise the CTA's partial (m, L and
// the unnormalised accumulators, fragment order) into workspace slot `slot`.
template <int KVT>
__device__ void merge_slots(const KParams &p, uint32_t base, int nsl, int mt, bool whole,
                            int row0, int head0, int slot, int ctid) {
  const int units = mt * 512;
  const int64_t per_slot = (int64_t)(p.mmax / kG) * 512;  // float4s per workspace slot
  for (int u = ctid; u < units; u += kNCW * 32) {
    const int mtile = u >> 9, rem = u & 511, i = rem >> 5, ln = rem & 31, g = ln >> 2, t = ln & 3;
    float M0 = -INFINITY, M1 = -INFINITY, L0 = 0.f, L1 = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 2
    for (int sl = 0; sl < nsl; ++sl) {
      const uint32_t sb = base + (sl * mt + mtile) * kSlotBytes;
      const uint4 a = lds128(sb + 8192 + ln * 16), b = lds128(sb + rem * 16);
      lse_combine(M0, M1, L0, L1, acc, __uint_as_float(a.x), __uint_as_float(a.y),
                  __uint_as_float(a.z), __uint_as_float(a.w),
                  make_float4(__uint_as_float(b.x), __uint_as_float(b.y), __uint_as_float(b.z),
                              __uint_as_float(b.w)));
    }
    if (whole) {
      const float s0 = L0 > 0.f ? p.vpost / L0 : 0.f, s1 = L1 > 0.f ? p.vpost / L1 : 0.f;
      store_unit<KVT>(p, row0 + mtile, head0, i, g, t, acc, s0, s1);
      if (i == 0 && t == 0 && p.lse != nullptr) {
        float *lp = p.lse + (int64_t)(row0 + mtile) * (p.Hkv * kG) + head0 + g;
        lp[0] = L0 > 0.f ? (M0 + log2f(L0)) * kLn2 : -INFINITY;
        lp[8] = L1 > 0.f ? (M1 + log2f(L1)) * kLn2 : -INFINITY;
      }
    } else {
      const int64_t ms = (int64_t)slot * (p.mmax / kG) + mtile;
      __stcg(reinterpret_cast<float4 *>(p.part_o) + (int64_t)slot * per_slot + mtile * 512 + rem, acc);
      if (i == 0 && t == 0)
        __stcg(reinterpret_cast<float4 *>(p.part_ml) + ms * 8 + g, make_float4(M0, M1, L0, L1));
    }
  }
}

// One share of a split sequence's merge, once every CTA of the sequence has stored its
// partial: CTA j of the sequence's nc CTAs merges float4 units [j U / nc, (j + 1) U / nc)
// of the U = q_len * 512 units of the output, G threads per unit (a power of two; each
// reads every G-th partial, then the G states combine through shuffles), so that every
// partial's load is in flight at once.
template <int KVT>
__device__ void merge_share(const KParams &p, int h, int row0, int qlen, int c_first, int nc,
                            int j, int ctid) {
  constexpr int kBatch = 4;  // partials per thread per memory round trip
  const int U = qlen * 512;
  const int u0 = (int)((int64_t)j * U / nc), u1 = (int)((int64_t)(j + 1) * U / nc);
  const int share = u1 - u0;
  int G = 1;
  while (G < 32 && G < nc && share * G * 2 <= kNCW * 32) G <<= 1;
  const float4 *po = reinterpret_cast<const float4 *>(p.part_o);
  const float4 *pml = reinterpret_cast<const float4 *>(p.part_ml);
  const int64_t per_slot = (int64_t)(p.mmax / kG) * 512;
  for (int q0 = 0; q0 < share * G; q0 += kNCW * 32) {
    const int q = q0 + ctid, uu = q / G, sub = q & (G - 1);
    const bool live = uu < share;
    const int u = u0 + (live ? uu : 0);
    const int mtile = u >> 9, rem = u & 511, i = rem >> 5, ln = rem & 31, g = ln >> 2, t = ln & 3;
    float M0 = -INFINITY, M1 = -INFINITY, L0 = 0.f, L1 = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (live) {
      for (int k0 = sub; k0 < nc; k0 += kBatch * G) {
        float4 ml[kBatch], x[kBatch];
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
          const int k = k0 + b * G;
          if (k < nc) {
            const int64_t sl = slot_of(c_first + k, c_first);
            ml[b] = __ldcg(pml + (sl * (p.mmax / kG) + mtile) * 8 + g);
            x[b] = __ldcg(po + sl * per_slot + mtile * 512 + rem);
          }
        }
#pragma unroll
        for (int b = 0; b < kBatch; ++b)
          if (k0 + b * G < nc) lse_combine(M0, M1, L0, L1, acc, ml[b].x, ml[b].y, ml[b].z, ml[b].w, x[b]);
      }
    }
    for (int o = 1; o < G; o <<= 1) {  // G | 32: the G threads of a unit sit in one warp
      const float m0 = __shfl_xor_sync(~0u, M0, o), m1 = __shfl_xor_sync(~0u, M1, o);
      const float l0 = __shfl_xor_sync(~0u, L0, o), l1 = __shfl_xor_sync(~0u, L1, o);
      float4 x;
      x.x = __shfl_xor_sync(~0u, acc.x, o);
      x.y = __shfl_xor_sync(~0u, acc.y, o);
      x.z = __shfl_xor_sync(~0u, acc.z, o);
      x.w = __shfl_xor_sync(~0u, acc.w, o);
      lse_combine(M0, M1, L0, L1, acc, m0, m1, l0, l1, x);
    }
    if (live && sub == 0) {
      const float s0 = L0 > 0.f ? p.vpost / L0 : 0.f, s1 = L1 > 0.f ? p.vpost / L1 : 0.f;
      store_unit<KVT>(p, row0 + mtile, h * kG, i, g, t, acc, s0, s1);
      if (i == 0 && t == 0 && p.lse != nullptr) {
        float *lp = p.lse + (int64_t)(row0 + mtile) * (p.Hkv * kG) + h * kG + g;
        lp[0] = L0 > 0.f ? (M0 + log2f(L0)) * kLn2 : -INFINITY;
        lp[8] = L1 > 0.f ? (M1 + log2f(L1)) * kLn2 : -INFINITY;
      }
    }
  }
}



}  // namespace pa
