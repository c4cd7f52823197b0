// pa_index.cu -- the indexer step before the sparse decode: pa_index_topk.
// See include/pa.h for the contract.
//
// Two launches.  index_score_kernel streams the e4m3 index cache once per request (a
// warp per page, a token per lane and 16 dimensions at a time, the request's index
// queries in shared memory as fp32) and writes each (row, page) score: the base-2
// log-sum-exp of the page's attended (head, token) scores.  index_select_kernel, a CTA
// per row, sorts that row's candidate pages by score in shared memory (bitonic, keys of
// score and page index) with the row's last attended page forced first, and writes the
// first topk.  HBM-bound on the index cache: 128 B per position per request.
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <cstdint>

#include "pa.h"

namespace {

constexpr int kD = 128;
constexpr int kWarps = 8;           // pages per CTA of the score kernel
constexpr int kMaxRowHeads = 16;    // q_len * index_heads of one request
constexpr int kMaxStride = 16384;   // pages per row the selection sorts
constexpr int kMaxTopk = 1024;

struct IdxParams {
  const uint16_t *q;
  const uint8_t *k;
  const float *ks;
  const int32_t *bt, *L, *cu;
  int32_t *sel, *nsel;
  float *scores;
  uint32_t *status;
  int64_t num_pages;
  int32_t B, R, H, ps, ps_shift, topk, stride, maxq;
  float cscale;  // sm_scale * log2(e)
};

__device__ __forceinline__ void e4m3x2_f32(uint32_t x, float &lo, float &hi) {
  asm("{\n\t.reg .b16 c, l, h;\n\t.reg .b32 w;\n\t"
      "cvt.u16.u32 c, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 w, c;\n\t"
      "mov.b32 {l, h}, w;\n\t"
      "cvt.f32.f16 %0, l;\n\t"
      "cvt.f32.f16 %1, h;\n\t}"
      : "=f"(lo), "=f"(hi)
      : "r"(x));
}

__device__ __forceinline__ uint4 load_nc16(const void *ptr) {
  uint4 r;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(ptr));
  return r;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Request blockIdx.y, pages blockIdx.x * kWarps + warp.  RH: q_len * index_heads rounded
// up to a power of two (rows past the request's are computed and dropped).
template <int RH>
__global__ void __launch_bounds__(kWarps * 32) index_score_kernel(const IdxParams p) {
  __shared__ float qs[RH * kD];
  const int r = blockIdx.y;
  const int L = p.L[r], row0 = p.cu[r], ql = p.cu[r + 1] - row0;
  if (ql < 0 || ql > p.maxq || L < ql || (int64_t)ql * p.H > RH || row0 < 0 || row0 + ql > p.R ||
      ((L + p.ps - 1) >> p.ps_shift) > p.stride) {
    if (threadIdx.x == 0 && blockIdx.x == 0 && p.status != nullptr)
      atomicOr(p.status, PA_DEV_BAD_INDEX_ROW);
    return;
  }
  if (ql == 0) return;
  const int npg = min((L + p.ps - 1) >> p.ps_shift, p.stride);
  if ((int)blockIdx.x * kWarps >= npg) return;  // the same for the whole CTA
  const int nrh = ql * p.H;
  for (int i = threadIdx.x; i < RH * kD; i += kWarps * 32)
    qs[i] = i < nrh * kD ? __uint_as_float((uint32_t)p.q[(int64_t)row0 * p.H * kD + i] << 16) : 0.f;
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.x * kWarps + warp;
  if (b >= npg) return;
  const int phys = p.bt[(int64_t)r * p.stride + b];
  if (phys < 0 || phys >= p.num_pages) {
    if (lane == 0 && p.status != nullptr) atomicOr(p.status, PA_DEV_BAD_PAGE);
    for (int t = lane; t < ql; t += 32) p.scores[(int64_t)(row0 + t) * p.stride + b] = -INFINITY;
    return;
  }
  // The lane's tokens t = lane + 32 i (i < 4, t < page_size), one at a time: a dot product
  // per (row, head) j, then a running (max, sum of 2^(s - max)) per j over the lane's
  // attended tokens; the warp combines them per row at the end.
  float m[RH], z[RH];
#pragma unroll
  for (int j = 0; j < RH; ++j) {
    m[j] = -INFINITY;
    z[j] = 0.f;
  }
  const uint8_t *kp = p.k + (int64_t)phys * p.ps * kD;
  const int pos0 = b * p.ps, lim_last = L;  // row ql-1 attends every position < L
#pragma unroll 1
  for (int i = 0; i < 4; ++i) {
    const int t = lane + 32 * i;
    if (t >= p.ps || pos0 + t >= lim_last) continue;  // no row attends it
    uint4 raw[kD / 16];
#pragma unroll
    for (int c = 0; c < kD / 16; ++c) raw[c] = load_nc16(kp + (int64_t)t * kD + c * 16);
    float acc[RH];
#pragma unroll
    for (int j = 0; j < RH; ++j) acc[j] = 0.f;
#pragma unroll
    for (int c = 0; c < kD / 16; ++c) {
      float kf[16];
      const uint32_t w[4] = {raw[c].x, raw[c].y, raw[c].z, raw[c].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        e4m3x2_f32(w[e] & 0xFFFFu, kf[4 * e + 0], kf[4 * e + 1]);
        e4m3x2_f32(w[e] >> 16, kf[4 * e + 2], kf[4 * e + 3]);
      }
#pragma unroll
      for (int j = 0; j < RH; ++j) {
        const float4 *q4 = reinterpret_cast<const float4 *>(qs + j * kD + c * 16);
        float a = acc[j];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float4 qv = q4[e];
          a = fmaf(qv.x, kf[4 * e + 0], a);
          a = fmaf(qv.y, kf[4 * e + 1], a);
          a = fmaf(qv.z, kf[4 * e + 2], a);
          a = fmaf(qv.w, kf[4 * e + 3], a);
        }
        acc[j] = a;
      }
    }
    const float sc = p.cscale * (p.ks != nullptr ? p.ks[(int64_t)phys * p.ps + t] : 1.f);
#pragma unroll
    for (int j = 0; j < RH; ++j) {
      if (j >= nrh) break;
      const int tok = j / p.H;
      if (pos0 + t >= L - ql + tok + 1) continue;  // past this row's cutoff
      const float sv = acc[j] * sc;
      if (sv > m[j]) {
        z[j] = z[j] * exp2f(m[j] - sv) + 1.f;
        m[j] = sv;
      } else {
        z[j] += exp2f(sv - m[j]);
      }
    }
  }
  for (int tok = 0; tok < ql; ++tok) {
    // the row's heads on this lane, then across the warp
    float mr = -INFINITY;
#pragma unroll
    for (int j = 0; j < RH; ++j)
      if (j / p.H == tok && j < nrh) mr = fmaxf(mr, m[j]);
    const float M = warp_max(mr);
    float zr = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int j = 0; j < RH; ++j)
        if (j / p.H == tok && j < nrh && m[j] != -INFINITY) zr += z[j] * exp2f(m[j] - M);
    }
    const float Z = warp_sum(zr);
    if (lane == 0)
      p.scores[(int64_t)(row0 + tok) * p.stride + b] = M == -INFINITY ? -INFINITY : M + log2f(Z);
  }
}

__device__ __forceinline__ uint32_t ordered_bits(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// A CTA per row; n (a power of two >= the row stride) keys in dynamic shared memory.
__global__ void __launch_bounds__(256) index_select_kernel(const IdxParams p, int n) {
  extern __shared__ unsigned long long keys[];
  const int row = blockIdx.x, tid = threadIdx.x;
  // the request that owns the row: the last r with cu[r] <= row
  int lo = 0, hi = p.B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.cu[mid] <= row)
      lo = mid;
    else
      hi = mid - 1;
  }
  const int r = lo, row0 = p.cu[r], ql = p.cu[r + 1] - row0, L = p.L[r];
  int nb = 0;
  if (row >= row0 && row < row0 + ql && ql <= p.maxq && L >= ql && row0 + ql <= p.R &&
      (int64_t)ql * p.H <= kMaxRowHeads && ((L + p.ps - 1) >> p.ps_shift) <= p.stride) {
    const int lim = L - ql + (row - row0) + 1;
    nb = lim > 0 ? min((lim + p.ps - 1) >> p.ps_shift, p.stride) : 0;
  }
  float *srow = p.scores + (int64_t)row * p.stride;
  for (int b = tid; b < n; b += 256) {
    unsigned long long k = 0ull;
    if (b < nb) {
      const uint32_t idx = 0xFFFFFFFFu - (uint32_t)b;
      k = b == nb - 1 ? ((0xFFFFFFFFull << 32) | idx)
                      : (((unsigned long long)ordered_bits(srow[b]) << 32) | idx);
    } else if (b < p.stride) {
      srow[b] = -INFINITY;
    }
    keys[b] = k;
  }
  __syncthreads();
  for (int k = 2; k <= n; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = tid; i < n; i += 256) {
        const int x = i ^ j;
        if (x > i) {
          const unsigned long long a = keys[i], c = keys[x];
          const bool desc = (i & k) == 0;
          if (desc ? a < c : a > c) {
            keys[i] = c;
            keys[x] = a;
          }
        }
      }
      __syncthreads();
    }
  }
  const int cnt = min(nb, p.topk);
  for (int i = tid; i < p.topk; i += 256)
    p.sel[(int64_t)row * p.topk + i] =
        i < cnt ? (int32_t)(0xFFFFFFFFu - (uint32_t)(keys[i] & 0xFFFFFFFFull)) : -1;
  if (tid == 0) p.nsel[row] = cnt;
}

bool aligned(const void *ptr, uintptr_t a) { return (reinterpret_cast<uintptr_t>(ptr) % a) == 0; }

int log2_page(int ps) {
  switch (ps) {
    case 16: return 4;
    case 32: return 5;
    case 64: return 6;
    case 128: return 7;
    default: return -1;
  }
}

template <int RH>
cudaError_t launch_scores(const IdxParams &p, int gx, cudaStream_t s) {
  index_score_kernel<RH><<<dim3(gx, p.B), kWarps * 32, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

extern "C" pa_status_t pa_index_topk(const pa_index_args_t *a, void *stream) {
  if (a == nullptr) return PA_ERR_INVALID_ARG;
  if (a->num_seqs < 1 || a->num_rows < 0 || a->index_heads < 1 || a->max_q_len < 1 ||
      a->num_pages < 1 || a->topk < 1 || a->topk > kMaxTopk || a->block_table_stride < 1 ||
      a->block_table_stride > kMaxStride || a->reserved != 0 || !(a->sm_scale > 0.f) ||
      !std::isfinite(a->sm_scale))
    return PA_ERR_INVALID_ARG;
  if (a->head_dim != kD) return PA_ERR_UNSUPPORTED;
  const int shift = log2_page(a->page_size);
  if (shift < 0) return PA_ERR_UNSUPPORTED;
  if ((int64_t)a->max_q_len * a->index_heads > kMaxRowHeads) return PA_ERR_UNSUPPORTED;
  if (a->num_pages > INT32_MAX) return PA_ERR_INVALID_ARG;
  if (a->q == nullptr || a->k_cache == nullptr || a->block_table == nullptr ||
      a->context_lens == nullptr || a->cu_seqlens_q == nullptr || a->selected == nullptr ||
      a->num_selected == nullptr || a->scores == nullptr)
    return PA_ERR_INVALID_ARG;
  if (!aligned(a->q, 16) || !aligned(a->k_cache, 16) || !aligned(a->scores, 16) ||
      (a->k_scale != nullptr && !aligned(a->k_scale, 4)) || !aligned(a->block_table, 4) ||
      !aligned(a->context_lens, 4) || !aligned(a->cu_seqlens_q, 4) || !aligned(a->selected, 4) ||
      !aligned(a->num_selected, 4) || (a->status != nullptr && !aligned(a->status, 4)))
    return PA_ERR_ALIGN;
  if (a->num_rows == 0) return PA_OK;

  IdxParams p;
  p.q = static_cast<const uint16_t *>(a->q);
  p.k = static_cast<const uint8_t *>(a->k_cache);
  p.ks = a->k_scale;
  p.bt = a->block_table;
  p.L = a->context_lens;
  p.cu = a->cu_seqlens_q;
  p.sel = a->selected;
  p.nsel = a->num_selected;
  p.scores = a->scores;
  p.status = a->status;
  p.num_pages = a->num_pages;
  p.B = a->num_seqs;
  p.R = a->num_rows;
  p.H = a->index_heads;
  p.ps = a->page_size;
  p.ps_shift = shift;
  p.topk = a->topk;
  p.stride = a->block_table_stride;
  p.maxq = a->max_q_len;
  p.cscale = a->sm_scale * 1.4426950408889634f;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int gx = (a->block_table_stride + kWarps - 1) / kWarps;
  const int rh = a->max_q_len * a->index_heads;
  cudaError_t e = rh <= 1   ? launch_scores<1>(p, gx, s)
                  : rh <= 2 ? launch_scores<2>(p, gx, s)
                  : rh <= 4 ? launch_scores<4>(p, gx, s)
                  : rh <= 8 ? launch_scores<8>(p, gx, s)
                            : launch_scores<16>(p, gx, s);
  if (e != cudaSuccess) return PA_ERR_CUDA;
  int n = 1;
  while (n < a->block_table_stride) n <<= 1;
  const size_t smem = (size_t)n * sizeof(unsigned long long);
  if (smem > 48 * 1024) {
    static bool opted = false;  // the kernel's opt-in limit, set once
    if (!opted) {
      if (cudaFuncSetAttribute(index_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)(kMaxStride * sizeof(unsigned long long))) != cudaSuccess)
        return PA_ERR_CUDA;
      opted = true;
    }
  }
  index_select_kernel<<<a->num_rows, 256, smem, s>>>(p, n);
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}
