// pa_index.cu -- the indexer step before the sparse decode: pa_index_topk.
// See include/pa.h for the contract.
//
// Two launches.  index_score_kernel streams the e4m3 index cache once per request (a
// warp per page; the request's index query rows against the page's tokens on the tensor
// cores, mma.sync m16n8k16 in f16 with fp32 accumulation) and writes each (row, page)
// score: the base-2 log-sum-exp of the page's attended (head, token) scores.  index_select_kernel, a CTA
// per row, sorts that row's candidate pages by score (bitonic, keys of score and page
// index; the stages within a warp on shuffles, the wider ones in shared memory) with the
// row's last attended page forced first, and writes the first topk.  HBM-bound on the index cache: 128 B per position per request.
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdint>
#include <mutex>

#include <cuda_fp16.h>

#include "pa.h"
#include "pa_ptx.cuh"

namespace {

constexpr int kD = 128;
constexpr int kWarps = 8;           // warps per CTA of the score kernel
constexpr int kMaxPagesPerWarp = 32;  // pages one warp of the score kernel scores (one per lane)
// A step of the score kernel: kStepTiles n-tiles (8 positions each) of one page, their
// codes and scales, staged through a ring of kSteps slots per warp with cp.async.
constexpr int kStepTiles = 4;
constexpr int kSteps = 3;
constexpr int kStepRows = 8 * kStepTiles;
constexpr int kStepBytes = (kStepRows * kD + kStepRows * 4 + 127) / 128 * 128;
static_assert(kStepRows <= 32, "a step's scales are one per lane");
constexpr int kRingBytes = kWarps * kSteps * kStepBytes;
constexpr int kQRow = 144;          // halves per staged query row (72 words)
constexpr int kMaxRowHeads = 16;    // q_len * index_heads of one request
constexpr int kMaxStride = 16384;   // pages per row the selection sorts
constexpr int kMaxTopk = 1024;
constexpr int kMaxDevices = 64;     // devices whose kernel opt-ins and SM count are tracked

// Asynchronous global -> shared copies of 16 bytes (through L2 only) and of 4 bytes; each
// thread tracks its own copies in commit groups.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void *src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// Waits until at most N of this thread's commit groups are still in flight.
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

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
  int32_t ppw;   // pages per warp of the score kernel: CTA x of a request scores pages
                 // [x kWarps ppw, (x + 1) kWarps ppw)
  float cscale;  // sm_scale * log2(e)
};

// Request blockIdx.y, pages blockIdx.x * kWarps + warp.  The request's q_len * heads
// query rows (at most 16, padded with zeros) are the M = 16 rows of mma.sync m16n8k16 in
// f16 (bf16 -> f16 is exact for 2^-14 <= |q| <= 65504); the page's tokens are the N
// columns, 8 per n-tile; its e4m3 codes widen exactly to f16.  The reduction index is
// permuted: in k-step kk, lane (g, t) supplies real dimensions 32 t + 4 kk + 0..3 for both
// operands, so each lane reads 32 contiguous bytes of a token row and the four lanes of a
// quad cover the whole 128-byte row.  Each warp streams its pages through its own ring of
// kSteps shared-memory slots with cp.async, two steps ahead of the one it computes (the
// 16-byte chunks of a row are XOR-swizzled by the row, so the quads' reads meet no bank
// conflict), which keeps twice the bytes of a register double buffer in flight.
__global__ void __launch_bounds__(kWarps * 32, 2) index_score_kernel(const IdxParams p) {
  extern __shared__ __align__(128) uint8_t ring[];
  // f16 query rows in k-step order: row, k-step kk, lane column t, then the 4 dimensions
  // 32 t + 4 kk + 0..3; rows 72 words apart so that a fragment load has no bank conflict
  __shared__ __align__(16) uint16_t qh[16 * kQRow];
  __shared__ float rowstat[kWarps][16][2];           // per warp: (max, sum) of each row
  const int r = blockIdx.y;
  const int L = p.L[r], row0 = p.cu[r], ql = p.cu[r + 1] - row0;
  if (ql < 0 || ql > p.maxq || L < ql || (int64_t)ql * p.H > 16 || row0 < 0 || row0 + ql > p.R ||
      ((L + p.ps - 1) >> p.ps_shift) > p.stride) {
    if (threadIdx.x == 0 && blockIdx.x == 0 && p.status != nullptr)
      atomicOr(p.status, PA_DEV_BAD_INDEX_ROW);
    return;
  }
  if (ql == 0) return;
  const int npg = min((L + p.ps - 1) >> p.ps_shift, p.stride);
  if ((int)blockIdx.x * kWarps * p.ppw >= npg) return;  // the same for the whole CTA
  const int nrh = ql * p.H;
  bool qbad = false;
  for (int i = threadIdx.x; i < 16 * kD; i += kWarps * 32) {
    float v = 0.f;
    if (i < nrh * kD) v = __uint_as_float((uint32_t)p.q[(int64_t)row0 * p.H * kD + i] << 16);
    qbad |= fabsf(v) > 65504.f;
    const int row = i / kD, d = i - row * kD;
    qh[row * kQRow + ((d & 31) >> 2) * 16 + (d >> 5) * 4 + (d & 3)] = __half_as_ushort(__float2half_rn(v));
  }
  if (qbad && p.status != nullptr) atomicOr(p.status, PA_DEV_Q_RANGE);
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  // this warp's pages: b_i = blockIdx.x * kWarps * ppw + warp + kWarps * i
  const int bfirst = blockIdx.x * kWarps * p.ppw + warp;
  int npw = 0;
  while (npw < p.ppw && bfirst + kWarps * npw < npg) ++npw;
  if (npw == 0) return;
  int my_phys = 0;  // lane i holds page i's physical page
  if (lane < npw) my_phys = p.bt[(int64_t)r * p.stride + bfirst + kWarps * lane];
  const bool my_bad = lane < npw && (my_phys < 0 || my_phys >= p.num_pages);
  if (__any_sync(0xffffffffu, my_bad) && lane == 0 && p.status != nullptr)
    atomicOr(p.status, PA_DEV_BAD_PAGE);
  // A fragments of k-step kk: rows g and g + 8 at dimensions 32 t + 4 kk + 0..3
  const uint16_t *qa = qh + g * kQRow + 4 * t, *qb = qh + (g + 8) * kQRow + 4 * t;
  uint32_t af[8][4];  // held for the warp's pages (reading them per k-step measured slower)
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const uint2 x = *reinterpret_cast<const uint2 *>(qa + 16 * kk);
    const uint2 y = *reinterpret_cast<const uint2 *>(qb + 16 * kk);
    af[kk][0] = x.x;
    af[kk][1] = y.x;
    af[kk][2] = x.y;
    af[kk][3] = y.y;
  }
  // rows g and g + 8: the cutoff of their query token (padding rows attend nothing)
  const int rowA = g, rowB = g + 8;
  const int limA = rowA < nrh ? L - ql + rowA / p.H + 1 : INT_MIN;
  const int limB = rowB < nrh ? L - ql + rowB / p.H + 1 : INT_MIN;
  const int ntiles = p.ps >> 3, ngr = (ntiles + kStepTiles - 1) / kStepTiles, total = npw * ngr;

  // step it: page it / ngr of the warp, n-tiles kStepTiles (it % ngr) onwards, into ring slot
  // `slot`
  const uint32_t wring = pa::smem_u32(ring) + warp * kSteps * kStepBytes;
  auto issue = [&](int it, int slot) {
    const int i = it / ngr, j0 = kStepTiles * (it - i * ngr);
    int ph = __shfl_sync(0xffffffffu, my_phys, i);
    const bool bad = __shfl_sync(0xffffffffu, my_bad ? 1 : 0, i) != 0;
    if (bad) ph = 0;  // read a valid page; the page's scores are written as -inf
    const int rows = min(kStepRows, p.ps - 8 * j0);
    const uint8_t *kp = p.k + ((int64_t)ph * p.ps + 8 * j0) * kD;
    const uint32_t sb = wring + slot * kStepBytes;
#pragma unroll
    for (int k = 0; k < kStepRows / 4; ++k) {
      const int q = lane + 32 * k, x = q >> 3, c = q & 7;  // row x, 16-byte chunk c
      if (x < rows) cp_async16(sb + x * kD + ((c ^ (x & 7)) << 4), kp + x * kD + 16 * c);
    }
    if (p.ks != nullptr && lane < rows)
      cp_async4(sb + kStepRows * kD + 4 * lane, p.ks + (int64_t)ph * p.ps + 8 * j0 + lane);
  };
  float mA = -INFINITY, zA = 0.f, mB = -INFINITY, zB = 0.f;
  // One step's scores of a row (this lane's 2 kStepTiles columns) into the row's running
  // (max, sum of 2^(s - max)): one maximum, one rescale and an exp2 per score, no branch;
  // masked positions enter as -inf.
  auto fold = [&](const float (&v)[2 * kStepTiles], float &m, float &z) {
    float mx = m;
#pragma unroll
    for (int k = 0; k < 2 * kStepTiles; ++k) mx = fmaxf(mx, v[k]);
    const float ref = mx == -INFINITY ? 0.f : mx;
    float sum = 0.f;
#pragma unroll
    for (int k = 0; k < 2 * kStepTiles; ++k) sum += pa::fast_exp2(v[k] - ref);
    z = z * pa::fast_exp2(m - ref) + sum;
    m = mx;
  };
  auto compute = [&](int it, int slot) {
    const int i = it / ngr, j0 = kStepTiles * (it - i * ngr);
    const int pos0 = (bfirst + kWarps * i) * p.ps;
    const uint32_t sb = wring + slot * kStepBytes;
    float vA[2 * kStepTiles], vB[2 * kStepTiles];
#pragma unroll
    for (int u = 0; u < kStepTiles; ++u) {
      const int j = j0 + u;
      vA[2 * u] = vA[2 * u + 1] = vB[2 * u] = vB[2 * u + 1] = -INFINITY;
      if (j >= ntiles) continue;
      const uint32_t rb = sb + (8 * u + g) * kD;
      const uint4 x0 = pa::lds128(rb + (((2 * t) ^ g) << 4));
      const uint4 x1 = pa::lds128(rb + (((2 * t + 1) ^ g) << 4));
      const uint32_t w[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        uint32_t b0, b1;
        pa::e4m3x4_to_f16x2x2(w[kk], b0, b1);
        pa::mma_f16(acc, af[kk], b0, b1);
      }
      const int tk = pos0 + 8 * j + 2 * t;
      float s0 = p.cscale, s1 = p.cscale;
      if (p.ks != nullptr) {
        const float2 kv = pa::lds64f(sb + kStepRows * kD + 4 * (8 * u + 2 * t));
        s0 *= kv.x;
        s1 *= kv.y;
      }
      vA[2 * u] = tk < limA ? acc[0] * s0 : -INFINITY;
      vA[2 * u + 1] = tk + 1 < limA ? acc[1] * s1 : -INFINITY;
      vB[2 * u] = tk < limB ? acc[2] * s0 : -INFINITY;
      vB[2 * u + 1] = tk + 1 < limB ? acc[3] * s1 : -INFINITY;
    }
    fold(vA, mA, zA);
    fold(vB, mB, zB);
  };
  auto finish = [&](int i) {  // page i of the warp: combine, write, reset
    const int bpage = bfirst + kWarps * i;
    const bool bad = __shfl_sync(0xffffffffu, my_bad ? 1 : 0, i) != 0;
#pragma unroll
    for (int o = 1; o <= 2; o <<= 1) {  // the quad's four lanes hold the same two rows
      const float m2A = __shfl_xor_sync(0xffffffffu, mA, o), z2A = __shfl_xor_sync(0xffffffffu, zA, o);
      const float m2B = __shfl_xor_sync(0xffffffffu, mB, o), z2B = __shfl_xor_sync(0xffffffffu, zB, o);
      const float nA = fmaxf(mA, m2A), nB = fmaxf(mB, m2B);
      zA = (nA == -INFINITY) ? 0.f : zA * pa::fast_exp2(mA - nA) + z2A * pa::fast_exp2(m2A - nA);
      zB = (nB == -INFINITY) ? 0.f : zB * pa::fast_exp2(mB - nB) + z2B * pa::fast_exp2(m2B - nB);
      mA = nA;
      mB = nB;
    }
    if (t == 0) {
      rowstat[warp][rowA][0] = mA;
      rowstat[warp][rowA][1] = zA;
      rowstat[warp][rowB][0] = mB;
      rowstat[warp][rowB][1] = zB;
    }
    __syncwarp();
    if (lane < ql) {  // query token `lane`: its heads' rows
      float M = -INFINITY;
      for (int h = 0; h < p.H; ++h) M = fmaxf(M, rowstat[warp][lane * p.H + h][0]);
      float Z = 0.f;
      if (M != -INFINITY)
        for (int h = 0; h < p.H; ++h) {
          const float mh = rowstat[warp][lane * p.H + h][0];
          if (mh != -INFINITY) Z += rowstat[warp][lane * p.H + h][1] * pa::fast_exp2(mh - M);
        }
      p.scores[(int64_t)(row0 + lane) * p.stride + bpage] =
          (bad || M == -INFINITY) ? -INFINITY : M + log2f(Z);
    }
    __syncwarp();
    mA = mB = -INFINITY;
    zA = zB = 0.f;
  };
  for (int it = 0; it < kSteps - 1; ++it) {
    if (it < total) issue(it, it);
    cp_async_commit();
  }
  for (int it = 0; it < total; ++it) {
    const int nx = it + kSteps - 1;  // refills the slot of step it - 1, read by now
    if (nx < total) issue(nx, nx % kSteps);
    cp_async_commit();
    cp_async_wait<kSteps - 1>();  // this lane's copies of step it have landed
    __syncwarp();                     // and so have the other lanes'
    compute(it, it % kSteps);
    if ((it + 1) % ngr == 0) finish(it / ngr);
    __syncwarp();  // every lane has read the slot before a later step refills it
  }
}

__device__ __forceinline__ uint32_t ordered_bits(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// A CTA per row; n (a power of two >= the row stride) keys in dynamic shared memory,
// sorted by a bitonic network whose every stage gives each thread one compare-exchange
// pair (up to 1024 threads).
__global__ void __launch_bounds__(1024) index_select_kernel(const IdxParams p, int n) {
  extern __shared__ unsigned long long keys[];
  const int row = blockIdx.x, tid = threadIdx.x, nt = blockDim.x;
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
  for (int b = tid; b < n; b += nt) {
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
  if (n == 2 * nt) {
    // Two keys per thread, elements 2 tid and 2 tid + 1, held in registers: the stages
    // whose pairs lie within a warp (distance j <= 32) run on shuffles with no barrier,
    // and only the wider ones (j >= 64) go through shared memory.
    unsigned long long x0 = keys[2 * tid], x1 = keys[2 * tid + 1];
    for (int k = 2; k <= n; k <<= 1) {
      int j = k >> 1;
      if (j >= 64) {
        keys[2 * tid] = x0;
        keys[2 * tid + 1] = x1;
        __syncthreads();
        for (; j >= 64; j >>= 1) {  // one pair per thread
          const int i = ((tid & ~(j - 1)) << 1) | (tid & (j - 1)), x = i + j;
          const unsigned long long a = keys[i], c = keys[x];
          const bool desc = (i & k) == 0;
          if (desc ? a < c : a > c) {
            keys[i] = c;
            keys[x] = a;
          }
          __syncthreads();
        }
        x0 = keys[2 * tid];
        x1 = keys[2 * tid + 1];
      }
      // elements e and e ^ j sit in lanes tid and tid ^ (j / 2); the pair's lower element
      // keeps the larger key in a descending block ((e & k) == 0), the smaller otherwise
      const bool desc = ((2 * tid) & k) == 0;
      for (; j >= 2; j >>= 1) {
        const unsigned long long y0 = __shfl_xor_sync(~0u, x0, j >> 1);
        const unsigned long long y1 = __shfl_xor_sync(~0u, x1, j >> 1);
        const bool takemax = (((2 * tid) & j) == 0) == desc;
        x0 = takemax ? (x0 > y0 ? x0 : y0) : (x0 < y0 ? x0 : y0);
        x1 = takemax ? (x1 > y1 ? x1 : y1) : (x1 < y1 ? x1 : y1);
      }
      const unsigned long long hi = x0 > x1 ? x0 : x1, lo = x0 > x1 ? x1 : x0;  // j = 1
      x0 = desc ? hi : lo;
      x1 = desc ? lo : hi;
    }
    keys[2 * tid] = x0;
    keys[2 * tid + 1] = x1;
    __syncthreads();
  } else {
    for (int k = 2; k <= n; k <<= 1) {
      for (int j = k >> 1; j > 0; j >>= 1) {
        for (int q = tid; q < (n >> 1); q += nt) {
          const int i = ((q & ~(j - 1)) << 1) | (q & (j - 1)), x = i + j;  // i has bit j clear
          const unsigned long long a = keys[i], c = keys[x];
          const bool desc = (i & k) == 0;
          if (desc ? a < c : a > c) {
            keys[i] = c;
            keys[x] = a;
          }
        }
        __syncthreads();
      }
    }
  }
  const int cnt = min(nb, p.topk);
  for (int i = tid; i < p.topk; i += nt)
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

int g_sms[kMaxDevices];  // SM count of each device, read with its opt-ins

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
  int dev = 0;
  int n = 1;
  while (n < a->block_table_stride) n <<= 1;
  const size_t smem = (size_t)n * sizeof(unsigned long long);
  {
    // the kernels' opt-in shared-memory limits, set once per device (the attributes
    // belong to the device's context)
    static std::once_flag once[kMaxDevices];
    static cudaError_t opt_err[kMaxDevices];
    if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return PA_ERR_UNSUPPORTED;
    std::call_once(once[dev], [dev]() {
      opt_err[dev] = cudaFuncSetAttribute(index_select_kernel,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          (int)(kMaxStride * sizeof(unsigned long long)));
      if (opt_err[dev] == cudaSuccess)
        opt_err[dev] = cudaFuncSetAttribute(index_score_kernel,
                                            cudaFuncAttributeMaxDynamicSharedMemorySize, kRingBytes);
      if (opt_err[dev] == cudaSuccess)
        opt_err[dev] = cudaDeviceGetAttribute(&g_sms[dev], cudaDevAttrMultiProcessorCount, dev);
    });
    if (opt_err[dev] != cudaSuccess) return PA_ERR_CUDA;
  }
  // One wave of score CTAs (two per SM): gx CTAs per request, each warp scoring ppw pages.
  const int stride = a->block_table_stride;
  int gx = std::max(1, 2 * g_sms[dev] / p.B);
  p.ppw = std::min(kMaxPagesPerWarp, (stride + kWarps * gx - 1) / (kWarps * gx));
  gx = (stride + kWarps * p.ppw - 1) / (kWarps * p.ppw);
  (void)cudaGetLastError();  // drop an earlier, unrelated launch error
  index_score_kernel<<<dim3(gx, p.B), kWarps * 32, kRingBytes, s>>>(p);
  if (cudaGetLastError() != cudaSuccess) return PA_ERR_CUDA;
  const int threads = n >= 2048 ? 1024 : (n >= 64 ? n / 2 : 32);
  index_select_kernel<<<a->num_rows, threads, smem, s>>>(p, n);
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}
