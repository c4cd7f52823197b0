// pa_kv_write.cu -- the producer of the per-token FP8 cache: pa_kv_quantize_write.
// See include/pa.h for the contract.
//
// HBM-bound: per (token, KV head) it reads 2 x 256 B of bf16 and writes 2 x (128 B of
// codes + a 4-B scale).  A warp takes four (token, head) units -- eight rows -- per step;
// each octet of lanes holds a row at a time, 16 values (32 B) per lane, and writes the
// row's 128 B of codes whole.  The loads of the next step are issued before the
// arithmetic of the current one, so two steps (4 KB) are in flight per warp.
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>

#include "pa.h"

namespace {

constexpr int kD = 128;
constexpr int kUnits = 4;          // (token, KV head) rows per warp step
constexpr int kWarps = 8;          // warps per CTA
constexpr float kE4m3Max = 448.f;  // largest finite e4m3fn value
constexpr bool kPipe = true;      // next step's loads before this step's arithmetic

struct KvWriteParams {
  const uint16_t *k_new, *v_new;
  const int64_t *slots;
  uint8_t *k_cache, *v_cache;
  float *k_scale, *v_scale;
  uint32_t *status;
  int64_t num_pages;
  int32_t units, Hkv, ps_shift;
};

// Four fp32 values -> four e4m3 codes (round to nearest even, saturating), first value
// in the lowest byte.
__device__ __forceinline__ uint32_t pack4_e4m3(float a, float b, float c, float d) {
  uint16_t lo, hi;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(b), "f"(a));
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(d), "f"(c));
  return (uint32_t)lo | ((uint32_t)hi << 16);
}

__device__ __forceinline__ uint4 load_nc16(const void *p) {
  uint4 r;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Codes of x[d] / s for 16 values: the e4m3 rounding (to nearest, ties to even, saturating
// at 448) of the exact quotient, s = fl(amax / 448) the stored scale.  Why one product is
// enough: with T = 448 x / amax (x, amax bf16: 8 significant bits each), 448 x - m amax is a
// multiple of a power of two for every rounding midpoint m (5 significant bits), so T is
// either exactly a midpoint or at least 2^-13 (relative) away from all of them; and x / s
// = T (amax / 448) / s lies within 2^-24 of T.  So a q within 2^-19 of x / s rounds like it,
// except where T is a midpoint: there x / s sits just below it when s was rounded up, just
// above when s was rounded down, and on it when s is exact -- the sign of 448 s - amax, one
// fma per row.  Hence q = x * A + x * B with, per row, r = 1/s rounded to nearest and
//   s rounded up or down: A = r (1 -+ 2^-20), B = 0: the bias pushes ties to the right side;
//   s exact: A = r, B = (1 - s r) r, the part of 1/s that r misses, so that q is x / s to
//     2^-47 and a tie lands on the midpoint itself, which the conversion rounds to even.
// Signs need nothing: the bias is relative and the conversion is symmetric.
__device__ __forceinline__ void encode_with(const float (&x)[16], float A, float B, float xs,
                                            uint32_t (&c)[4]) {
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    float q[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float a = x[4 * w + k] * xs;
      q[k] = fmaf(a, A, a * B);
    }
    c[w] = pack4_e4m3(q[0], q[1], q[2], q[3]);
  }
}

__device__ __forceinline__ void encode_scaled(const float (&x)[16], float amax, float s, float xs,
                                              uint32_t (&c)[4]) {
  const float r = __frcp_rn(s);
  const float side = fmaf(s, kE4m3Max, -amax);  // its sign is exact: 448 s - amax
  float A = r, B = 0.f;
  if (side > 0.f)
    A = r * (1.f - 0x1p-20f);
  else if (side < 0.f)
    A = r * (1.f + 0x1p-20f);
  else
    B = fmaf(-s, r, 1.f) * r;
  encode_with(x, A, B, xs, c);
}

__device__ __forceinline__ void encode_row(const float (&x)[16], float amax, float scale,
                                           uint32_t (&c)[4]) {
  if (scale < 0x1p-100f)  // keep 1 / s finite: x, amax and s times 2^100, exactly
    encode_scaled(x, amax * 0x1p100f, scale * 0x1p100f, 0x1p100f, c);
  else
    encode_scaled(x, amax, scale, 1.f, c);
}

// One warp step covers kUnits (token, KV head) units, i.e. 2 kUnits rows (K and V).  Lane
// octet o (lanes 8o .. 8o+7) takes rows o, o + 4, ...: row r is unit r / 2, K if r is even,
// and each lane holds 16 of the row's values (32 bytes).
constexpr int kRowsPerOctet = 2 * kUnits / 4;

struct Step {
  int64_t slot[kRowsPerOctet];
  uint4 raw[kRowsPerOctet][2];
};

__device__ __forceinline__ void load_step(const KvWriteParams &p, int grp, int oct, int l8,
                                          Step &st) {
#pragma unroll
  for (int j = 0; j < kRowsPerOctet; ++j) {
    const int r = oct + 4 * j, u = grp * kUnits + (r >> 1);
    const uint16_t *src = (r & 1) ? p.v_new : p.k_new;
    st.slot[j] = -1;
    st.raw[j][0] = st.raw[j][1] = make_uint4(0, 0, 0, 0);
    if (u < p.units) {
      st.slot[j] = __ldg(p.slots + (p.Hkv == 1 ? u : u / p.Hkv));
      const uint16_t *q = src + (int64_t)u * kD + l8 * 16;
      st.raw[j][0] = load_nc16(q);
      st.raw[j][1] = load_nc16(q + 8);
    }
  }
}

__device__ __forceinline__ void quantize_step(const KvWriteParams &p, const Step &st, int grp,
                                              int oct, int l8, int64_t nslots) {
#pragma unroll
  for (int j = 0; j < kRowsPerOctet; ++j) {
    const int r = oct + 4 * j, u = grp * kUnits + (r >> 1);
    const int64_t slot = st.slot[j];
    const bool live = slot >= 0 && slot < nslots;
    if (slot >= nslots && l8 == 0 && p.status != nullptr) atomicOr(p.status, PA_DEV_BAD_SLOT);
    float x[16];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint4 w = st.raw[j][h];
      x[8 * h + 0] = bf16_lo(w.x);
      x[8 * h + 1] = bf16_hi(w.x);
      x[8 * h + 2] = bf16_lo(w.y);
      x[8 * h + 3] = bf16_hi(w.y);
      x[8 * h + 4] = bf16_lo(w.z);
      x[8 * h + 5] = bf16_hi(w.z);
      x[8 * h + 6] = bf16_lo(w.w);
      x[8 * h + 7] = bf16_hi(w.w);
    }
    float amax = 0.f;
#pragma unroll
    for (int d = 0; d < 16; ++d) amax = fmaxf(amax, fabsf(x[d]));
#pragma unroll
    for (int o = 4; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    // scale = amax / 448, rounded once to fp32, is stored; each code is the e4m3 rounding
    // of the exact quotient x / scale.
    const float scale = __fdiv_rn(amax, kE4m3Max);
    uint4 codes = make_uint4(0, 0, 0, 0);
    if (scale != 0.f) {
      uint32_t c[4];
      encode_row(x, amax, scale, c);
      codes = make_uint4(c[0], c[1], c[2], c[3]);
    }
    if (!live) continue;
    const int head = p.Hkv == 1 ? 0 : u % p.Hkv;
    const int64_t pg = slot >> p.ps_shift, off = slot & ((1 << p.ps_shift) - 1);
    const int64_t row = ((pg * p.Hkv + head) << p.ps_shift) + off;
    uint8_t *cache = (r & 1) ? p.v_cache : p.k_cache;
    *reinterpret_cast<uint4 *>(cache + row * kD + l8 * 16) = codes;
    if (l8 == 0) ((r & 1) ? p.v_scale : p.k_scale)[row] = scale;
  }
}

template <bool PIPE>
__global__ void __launch_bounds__(kWarps * 32) kv_quantize_write_kernel(const KvWriteParams p) {
  const int lane = threadIdx.x & 31, oct = lane >> 3, l8 = lane & 7;
  const int ngroups = (p.units + kUnits - 1) / kUnits;
  const int nwarps = gridDim.x * kWarps;
  const int64_t nslots = p.num_pages << p.ps_shift;
  int grp = blockIdx.x * kWarps + (threadIdx.x >> 5);
  if (PIPE) {
    Step cur, nxt;
    if (grp < ngroups) load_step(p, grp, oct, l8, cur);
    for (; grp < ngroups; grp += nwarps) {
      // the next step's loads go out before this step's arithmetic
      if (grp + nwarps < ngroups) load_step(p, grp + nwarps, oct, l8, nxt);
      quantize_step(p, cur, grp, oct, l8, nslots);
      cur = nxt;
    }
  } else {
    for (; grp < ngroups; grp += nwarps) {
      Step cur;
      load_step(p, grp, oct, l8, cur);
      quantize_step(p, cur, grp, oct, l8, nslots);
    }
  }
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

}  // namespace

extern "C" pa_status_t pa_kv_quantize_write(const pa_kv_write_args_t *a, void *stream) {
  if (a == nullptr) return PA_ERR_INVALID_ARG;
  if (a->num_tokens < 0 || a->num_kv_heads < 1 || a->num_pages < 1 || a->reserved != 0)
    return PA_ERR_INVALID_ARG;
  if (a->head_dim != kD) return PA_ERR_UNSUPPORTED;
  const int shift = log2_page(a->page_size);
  if (shift < 0) return PA_ERR_UNSUPPORTED;
  if (a->num_tokens * (int64_t)a->num_kv_heads > INT_MAX) return PA_ERR_INVALID_ARG;
  if (a->num_pages > (INT64_MAX >> 16) / a->num_kv_heads) return PA_ERR_INVALID_ARG;
  if (a->k_new == nullptr || a->v_new == nullptr || a->slot_mapping == nullptr ||
      a->k_cache == nullptr || a->v_cache == nullptr || a->k_scale == nullptr ||
      a->v_scale == nullptr)
    return PA_ERR_INVALID_ARG;
  if (!aligned(a->k_new, 16) || !aligned(a->v_new, 16) || !aligned(a->k_cache, 16) ||
      !aligned(a->v_cache, 16) || !aligned(a->k_scale, 4) || !aligned(a->v_scale, 4) ||
      !aligned(a->slot_mapping, 8) || (a->status != nullptr && !aligned(a->status, 4)))
    return PA_ERR_ALIGN;
  if (a->num_tokens == 0) return PA_OK;

  KvWriteParams p;
  p.k_new = static_cast<const uint16_t *>(a->k_new);
  p.v_new = static_cast<const uint16_t *>(a->v_new);
  p.slots = a->slot_mapping;
  p.k_cache = static_cast<uint8_t *>(a->k_cache);
  p.v_cache = static_cast<uint8_t *>(a->v_cache);
  p.k_scale = a->k_scale;
  p.v_scale = a->v_scale;
  p.status = a->status;
  p.num_pages = a->num_pages;
  p.units = (int32_t)(a->num_tokens * a->num_kv_heads);
  p.Hkv = a->num_kv_heads;
  p.ps_shift = shift;

  // SMs and resident CTAs per SM, looked up once per device
  static int cached[64][2];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
  int sms = 0, per_sm = 0;
  if (dev >= 0 && dev < 64 && cached[dev][0] > 0) {
    sms = cached[dev][0];
    per_sm = cached[dev][1];
  } else {
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kv_quantize_write_kernel<kPipe>,
                                                      kWarps * 32, 0) != cudaSuccess)
      return PA_ERR_CUDA;
    if (dev >= 0 && dev < 64) {
      cached[dev][1] = per_sm;
      cached[dev][0] = sms;
    }
  }
  const int64_t groups = (p.units + kUnits - 1) / kUnits;
  const int64_t want = (groups + kWarps - 1) / kWarps;
  const int64_t cap = (int64_t)sms * (per_sm > 0 ? per_sm : 1);  // one wave of resident CTAs
  const int grid = (int)(want < cap ? want : cap);
  (void)cudaGetLastError();  // drop an earlier, unrelated launch error
  kv_quantize_write_kernel<kPipe><<<grid, kWarps * 32, 0, static_cast<cudaStream_t>(stream)>>>(p);
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}
