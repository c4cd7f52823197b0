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

#include "pa_kernel.cuh"

namespace pa {

struct Frag {
  uint32_t qf[8][4];
  float o[16][4];
  float m[2], l[2];
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
}

// ------------------------------------------------------------------------ online softmax

// s holds the log2-domain scores of this lane's 4 columns of one row; on return it
// holds p = 2^(s - m) with m the row's running maximum.  Rescales l and the row's
// accumulators (o[.][half], o[.][half + 1]) when the maximum grows.
__device__ __forceinline__ void online_row(float (&s)[4], float &m, float &l, float (&o)[16][4],
                                           int half) {
  float mx = fmaxf(fmaxf(s[0], s[1]), fmaxf(s[2], s[3]));
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
  for (int k = 0; k < 4; ++k) s[k] = fast_exp2(s[k] - ref);
  l += (s[0] + s[1]) + (s[2] + s[3]);
}

// Scores of the 4 columns of rows g (s0) and g + 8 (s1) -> masked -> softmax update.
// pos0 is the position of token 2t of the chunk (or < 0 when the page slot is empty).
__device__ __forceinline__ void mask_scores(float (&s0)[4], float (&s1)[4], int pos0, int cut) {
  const int off[4] = {0, 1, 8, 9};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    if (pos0 < 0 || pos0 + off[k] >= cut) {
      s0[k] = -INFINITY;
      s1[k] = -INFINITY;
    }
  }
}

// --------------------------------------------------------------------- one 16-token chunk

// FP8 tile: K at st, V at st + 16384 (each [128 tokens][128 B], 128-byte swizzle),
// K scales at st + 32768, V scales at st + 33280 (fp32 per token).
template <int SM>
__device__ __forceinline__ void chunk_fp8(const KParams &p, uint32_t st, int tb, bool masked,
                                          int pos0, int cut, int g, int t, Frag &f) {
  const uint32_t Kb = st, Vb = st + 16384;
  const uint32_t sw0 = ((2 * t) ^ g) << 4, sw1 = ((2 * t + 1) ^ g) << 4;
  const uint4 ka0 = lds128(Kb + (tb + g) * 128 + sw0), ka1 = lds128(Kb + (tb + g) * 128 + sw1);
  const uint4 kb0 = lds128(Kb + (tb + 8 + g) * 128 + sw0);
  const uint4 kb1 = lds128(Kb + (tb + 8 + g) * 128 + sw1);
  const uint32_t wa[8] = {ka0.x, ka0.y, ka0.z, ka0.w, ka1.x, ka1.y, ka1.z, ka1.w};
  const uint32_t wb[8] = {kb0.x, kb0.y, kb0.z, kb0.w, kb1.x, kb1.y, kb1.z, kb1.w};
  float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    uint32_t b0, b1, c0, c1;
    e4m3x4_to_f16x2x2(wa[kk], b0, b1);
    e4m3x4_to_f16x2x2(wb[kk], c0, c1);
    mma_f16(sa, f.qf[kk], b0, b1);
    mma_f16(sb, f.qf[kk], c0, c1);
  }
  float k0, k1, k2, k3;
  if (SM == PA_SCALE_PER_TOKEN) {
    const float2 x = lds64f(st + 32768 + (tb + 2 * t) * 4);
    const float2 y = lds64f(st + 32768 + (tb + 8 + 2 * t) * 4);
    k0 = x.x * p.kfold;
    k1 = x.y * p.kfold;
    k2 = y.x * p.kfold;
    k3 = y.y * p.kfold;
  } else {
    k0 = k1 = k2 = k3 = p.kfold;
  }
  float s0[4] = {sa[0] * k0, sa[1] * k1, sb[0] * k2, sb[1] * k3};
  float s1[4] = {sa[2] * k0, sa[3] * k1, sb[2] * k2, sb[3] * k3};
  if (masked) mask_scores(s0, s1, pos0, cut);
  online_row(s0, f.m[0], f.l[0], f.o, 0);
  online_row(s1, f.m[1], f.l[1], f.o, 2);
  uint32_t pa[4];
  if (SM == PA_SCALE_PER_TOKEN) {
    const float2 x = lds64f(st + 33280 + (tb + 2 * t) * 4);
    const float2 y = lds64f(st + 33280 + (tb + 8 + 2 * t) * 4);
    const float w0 = x.x * p.pfold, w1 = x.y * p.pfold, w2 = y.x * p.pfold, w3 = y.y * p.pfold;
    pa[0] = pack_f16x2(s0[0] * w0, s0[1] * w1);
    pa[1] = pack_f16x2(s1[0] * w0, s1[1] * w1);
    pa[2] = pack_f16x2(s0[2] * w2, s0[3] * w3);
    pa[3] = pack_f16x2(s1[2] * w2, s1[3] * w3);
  } else {
    pa[0] = pack_f16x2(s0[0], s0[1]);
    pa[1] = pack_f16x2(s1[0], s1[1]);
    pa[2] = pack_f16x2(s0[2], s0[3]);
    pa[3] = pack_f16x2(s1[2], s1[3]);
  }
  const int rv = tb + 2 * t;
  const uint32_t sv0 = (g ^ (2 * t)) << 4, sv1 = (g ^ (2 * t + 1)) << 4;
  const uint4 va = lds128(Vb + rv * 128 + sv0), vb = lds128(Vb + (rv + 1) * 128 + sv1);
  const uint4 vc = lds128(Vb + (rv + 8) * 128 + sv0), vd = lds128(Vb + (rv + 9) * 128 + sv1);
  const uint32_t A[4] = {va.x, va.y, va.z, va.w}, Bw[4] = {vb.x, vb.y, vb.z, vb.w};
  const uint32_t C[4] = {vc.x, vc.y, vc.z, vc.w}, Dw[4] = {vd.x, vd.y, vd.z, vd.w};
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    uint32_t x0, x1, y0, y1;
    e4m3x4_to_f16x2x2(prmt(A[w], Bw[w], 0x5140), x0, x1);
    e4m3x4_to_f16x2x2(prmt(C[w], Dw[w], 0x5140), y0, y1);
    mma_f16(f.o[4 * w], pa, x0, y0);
    mma_f16(f.o[4 * w + 1], pa, x1, y1);
    e4m3x4_to_f16x2x2(prmt(A[w], Bw[w], 0x7362), x0, x1);
    e4m3x4_to_f16x2x2(prmt(C[w], Dw[w], 0x7362), y0, y1);
    mma_f16(f.o[4 * w + 2], pa, x0, y0);
    mma_f16(f.o[4 * w + 3], pa, x1, y1);
  }
}

// BF16 tile: K halves (d 0-63, 64-127) at st and st + 16384, V halves at st + 32768 and
// st + 49152, each [128 tokens][128 B] with 128-byte swizzle.
__device__ __forceinline__ void chunk_bf16(const KParams &p, uint32_t st, int tb, bool masked,
                                           int pos0, int cut, int g, int t, int lane, Frag &f) {
  const int mat = lane >> 3, rr = lane & 7;
  float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
  {
    const int row = tb + 8 * (mat >> 1) + rr;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const int c16 = 2 * kk + (mat & 1);
      const uint32_t addr = st + (c16 >> 3) * 16384 + row * 128 + (((c16 & 7) ^ rr) << 4);
      uint32_t r0, r1, r2, r3;
      ldsm_x4(addr, r0, r1, r2, r3);
      mma_bf16(sa, f.qf[kk], r0, r1);
      mma_bf16(sb, f.qf[kk], r2, r3);
    }
  }
  const float k = p.kfold;
  float s0[4] = {sa[0] * k, sa[1] * k, sb[0] * k, sb[1] * k};
  float s1[4] = {sa[2] * k, sa[3] * k, sb[2] * k, sb[3] * k};
  if (masked) mask_scores(s0, s1, pos0, cut);
  online_row(s0, f.m[0], f.l[0], f.o, 0);
  online_row(s1, f.m[1], f.l[1], f.o, 2);
  uint32_t pa[4];
  pa[0] = pack_bf16x2(s0[0], s0[1]);
  pa[1] = pack_bf16x2(s1[0], s1[1]);
  pa[2] = pack_bf16x2(s0[2], s0[3]);
  pa[3] = pack_bf16x2(s1[2], s1[3]);
  const int tok = tb + 8 * (mat & 1) + rr;
#pragma unroll
  for (int j = 0; j < 16; j += 2) {
    const int c16 = j + (mat >> 1);
    const uint32_t addr = st + 32768 + (c16 >> 3) * 16384 + tok * 128 + (((c16 & 7) ^ rr) << 4);
    uint32_t r0, r1, r2, r3;
    ldsm_x4_t(addr, r0, r1, r2, r3);
    mma_bf16(f.o[j], pa, r0, r1);
    mma_bf16(f.o[j + 1], pa, r2, r3);
  }
}

// ------------------------------------------------------------------------ state exchange

// Merge-buffer slot k: accumulators as [16][32 lanes][4] floats, then m0, m1, l0, l1.
__device__ __forceinline__ void put_state(const Smem &sm, int k, const Frag &f, int lane) {
  const uint32_t ob = sm.merge() + k * 8192, mb = sm.merge() + 32768 + k * 512;
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
  const uint32_t ob = sm.merge() + k * 8192, mb = sm.merge() + 32768 + k * 512;
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

// Split-K partial of one m-tile: m, l per row and the unnormalised o in natural d order.
template <int KVT>
__device__ __forceinline__ void write_partial(const KParams &p, const Frag &f, int slot,
                                              int mtile, int g, int t) {
#pragma unroll
  for (int hf = 0; hf < 2; ++hf) {
    const float lq = quad_sum(f.l[hf]);
    const int rowi = mtile * kG + g + 8 * hf;
    if (t == 0) {
      p.part_ml[((int64_t)slot * 2) * p.mmax + rowi] = f.m[hf];
      p.part_ml[((int64_t)slot * 2 + 1) * p.mmax + rowi] = lq;
    }
    float *dst = p.part_o + ((int64_t)slot * p.mmax + rowi) * kD;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      dst[dmap<KVT>(i, 0, t)] = f.o[i][2 * hf];
      dst[dmap<KVT>(i, 1, t)] = f.o[i][2 * hf + 1];
    }
  }
}

// The last CTA to finish a split sequence merges every partial (log-sum-exp merge).
__device__ void merge_partials(const KParams &p, int r, int h, int row0, int qlen, int c_first,
                               int n, int ctid) {
  const int rows = qlen * kG, Hq = p.Hkv * kG;
  for (int u = ctid; u < rows * 32; u += kNCW * 32) {
    const int row = u >> 5, d4 = u & 31;
    float M = -INFINITY;
    for (int k = 0; k < n; ++k) {
      const int sl = slot_of(c_first + k, c_first);
      M = fmaxf(M, __ldcg(p.part_ml + ((int64_t)sl * 2) * p.mmax + row));
    }
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float Ls = 0.f;
    for (int k = 0; k < n; ++k) {
      const int sl = slot_of(c_first + k, c_first);
      const float mm = __ldcg(p.part_ml + ((int64_t)sl * 2) * p.mmax + row);
      const float w = (mm == -INFINITY) ? 0.f : fast_exp2(mm - M);
      Ls += w * __ldcg(p.part_ml + ((int64_t)sl * 2 + 1) * p.mmax + row);
      const float4 v = __ldcg(reinterpret_cast<const float4 *>(p.part_o + ((int64_t)sl * p.mmax + row) * kD) + d4);
      acc.x += w * v.x;
      acc.y += w * v.y;
      acc.z += w * v.z;
      acc.w += w * v.w;
    }
    const float sc = Ls > 0.f ? p.vpost / Ls : 0.f;
    const float v[4] = {acc.x * sc, acc.y * sc, acc.z * sc, acc.w * sc};
    const int orow = row0 + (row >> 4), head = h * kG + (row & 15);
    store_out(p, ((int64_t)orow * Hq + head) * kD + 4 * d4, v, 4);
    if (d4 == 0 && p.lse != nullptr)
      p.lse[(int64_t)orow * Hq + head] = Ls > 0.f ? (M + log2f(Ls)) * kLn2 : -INFINITY;
  }
}

}  // namespace pa
