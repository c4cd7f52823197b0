// pa_kernel.cuh -- the paged decode attention kernel for sm_103a.
//
// One persistent CTA per SM (balanced schedule) or one CTA per fixed split-K partition.
// Work is a list of KV tiles of 128 tokens: request-major, then KV head, then tile.
// Dense tiles cover positions [128 t, 128 t + 128); sparse tiles cover 128 / page_size
// consecutive entries of the request's selected-page list (ROCm/ATOM PR 2614,
// "Change": sparse decode reuses the dense paged-decode contract).
//
// Warp roles in a CTA of 9 warps:
//   warp 8     producer: walks the CTA's tile range, reads block-table (and selected-
//              page) entries, and moves each page's K and V rows into a shared-memory
//              stage with TMA (128-byte swizzle) plus the per-token scales and, at the
//              start of a request, the request's query rows, all completing on the
//              stage's mbarrier.
//   warps 0-7  consumers: exact e4m3 -> f16 widening in registers, QK^T and PV on
//              mma.sync tensor-core fragments, online softmax with warp shuffles,
//              per-token K scale folded into the score column and V scale into P
//              (vLLM PR 52060, "Suggested Fix"), a log-sum-exp merge across warps,
//              and, when a request spans several CTAs, split-K partials merged by the
//              last CTA to finish (ROCm/ATOM PR 2710 review, "Smaller": exp_sums,
//              max_logits, temporary_output).
// Every wait is bounded; a wait that gives up sets PA_DEV_TIMEOUT and the CTA drains.
#pragma once

#include <cstdint>
#include <cuda.h>

#include "pa.h"
#include "pa_ptx.cuh"

namespace pa {

// Launch trace (compiled in only with PA_TRACE): the global timer at fixed points of each
// CTA's run, kept for the last kTraceCalls launches of every CTA (slot = the CTA's launch
// count modulo kTraceCalls).  pa_debug_trace copies it out.  Without PA_TRACE the marks
// are empty functions.
enum : int {
  T_ENTRY = 0, T_PROLOGUE = 1, T_PRODUCER = 2, T_CONSUMER = 3, T_FIRST_TILE = 4,
  T_LAST_TILE = 5, T_STORED = 6, T_ARRIVED = 7, T_MERGE = 8, T_MERGED = 9, T_EXIT = 10,
  T_CALL = 11, T_A = 12, T_B = 13, T_LAST = 14, T_MARKS = 16
};
constexpr int kTraceCalls = 16, kTraceCtas = 1024;
#ifdef PA_TRACE
__device__ unsigned long long g_trace[kTraceCalls][kTraceCtas][T_MARKS];
__device__ unsigned int g_trace_count[kTraceCtas];
__device__ __forceinline__ void trace_value(int k, unsigned long long v) {
  if (blockIdx.x < kTraceCtas) g_trace[g_trace_count[blockIdx.x] % kTraceCalls][blockIdx.x][k] = v;
}
__device__ __forceinline__ void trace(int k) {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  trace_value(k, t);
}
// Ends this CTA's record of the launch (one thread, last).
__device__ __forceinline__ void trace_close() {
  if (blockIdx.x < kTraceCtas) {
    trace_value(T_CALL, g_trace_count[blockIdx.x]);
    trace(T_EXIT);
    ++g_trace_count[blockIdx.x];
  }
}
#else
__device__ __forceinline__ void trace_value(int, unsigned long long) {}
__device__ __forceinline__ void trace(int) {}
__device__ __forceinline__ void trace_close() {}
#endif

}  // namespace pa

namespace pa {

constexpr int kD = 128;          // head_dim
constexpr int kG = 16;           // query heads per KV head (rows of one m-tile)
constexpr int kTile = 128;       // tokens per KV tile
constexpr int kNCW = 8;          // consumer warps (two warpgroups)
constexpr int kThreads = (kNCW + 4) * 32;  // + one producer warpgroup (warp kNCW copies)
// Register split: the CTA is launched at kLaunchRegs per thread; the producer warpgroup
// gives registers back down to kProdRegs and the consumer warpgroups take kConsRegs.
// Both totals agree, per CTA and per SM sub-partition (each holds one warp of each
// warpgroup), so the consumers' increase is always satisfied.  The host refuses to
// launch a build whose register count is not kLaunchRegs.
constexpr int kLaunchRegs = 168, kProdRegs = 56, kConsRegs = 224;
static_assert(kNCW * 32 * kConsRegs + 4 * 32 * kProdRegs == kThreads * kLaunchRegs,
              "register split must match the launch allocation");
constexpr int kMaxQ = 8;         // most query tokens per request (m-tiles)
// End of a CTA's last sequence: its token slices merge in stage memory in one step (true)
// or pair through the exchange buffer (false).  A sequence split across co-resident CTAs:
// every one of them merges a share of it (true), or the last to arrive merges it (false).
constexpr bool kSlotMerge = true, kShareMerge = true;
// A shared merge needs this many partial m-tiles (CTAs x query tokens) of the sequence;
// smaller ones are merged by the last CTA to arrive.
constexpr int kShareMin = 8;
constexpr int kQRowBytes = kG * kD * 2;   // one query token's 16 heads, bf16
constexpr int kMergeBytes = 4 * 8192 + 4 * 512;  // the exchange buffer at 4 slots
constexpr int kUmmaBars = 24;    // extra mbarriers of the tcgen05 kernel
constexpr int kDumpHeader = 128;
constexpr float kLn2 = 0.693147180559945309f;

enum : int { F_BEGIN = 1, F_END = 2, F_MASK = 4, F_WHOLE = 8 };

// Written by the producer before it arrives on the stage's full barrier.
struct StageMeta {
  int32_t r, h, tile, flags;
  int32_t L, qlen, row0, nvalid;
  int32_t page_pos[8];   // first position of each page slot of the tile, -1 = empty
  int32_t page_phys[8];  // its physical page, -1 = empty
  int32_t gtile, qslot, pad[6];
};
static_assert(sizeof(StageMeta) == 128, "meta size");

struct KParams {
  CUtensorMap tm_k;               // 2-D map over [num_pages * Hkv * page_size rows, row bytes]
  CUtensorMap tm_v;
  const uint16_t *q;
  const uint8_t *k_cache, *v_cache;  // for the L2 prefetch of the first pages (before the wait)
  const float *k_scale, *v_scale;
  const int32_t *block_table, *context_lens, *cu_q, *sel, *nsel;
  void *out;
  float *lse;
  uint32_t *status;
  int32_t *counters;              // [num_seqs * Hkv] arrivals of split-K partials
  int32_t *flags;                 // [num_seqs * Hkv] generation of each sequence's merge (bumped by
                                  // the last arrival; the other CTAs wait for the bump)
  float *part_ml;                 // [slots][2][mmax]  (m in log2 units, l)
  float *part_o;                  // [slots][mmax][128] (unnormalised)
  uint8_t *dump;
  int64_t dump_tiles;
  int64_t num_pages;
  float kfold;                    // score = acc * kfold (* k_scale[token] in per-token mode)
  float pfold;                    // unused (1): the per-token V scale's power of two is per warp
  float vpost;                    // out = (o / l) * vpost
  int32_t num_seqs, Hkv, ps, ps_shift, ppt, bt_stride, sel_stride, q_uniform, max_q, max_ctx;
  int32_t num_rows, out_f32, sched_partition, part_tiles, maxch, grid, nstage, mmax, sparse;
  int32_t off_q, qslot_bytes, off_merge, off_tstart, off_meta, off_bar, off_misc, stage_bytes;
  int32_t xslots;                 // slots of the exchange buffer (4, or 2 for one-token FP8 plans)
  int32_t coresident;             // every CTA of the grid is resident at once (one per SM): the
                                  // CTAs of a split sequence may wait for each other and share
                                  // its merge; otherwise the last arrival merges it alone
};

// misc[] words
// M_LAST, M_LAST + 1: merge duty for the head / tail sequence; M_WCNT: writer warps that
// have stored their part of the head partial; M_WSUM..: 12 warp sums of the prologue scan.
// M_HEAD, M_TAIL: (request, head, first row, q_len, first CTA, CTA count) of each.
// M_TMEM: TMEM base address of the tcgen05 kernel.  M_ZERO: a 16-byte line of zeros.
// M_QHDR: (request, KV head, q_len, first row, context) of the request whose query sits
// in query slot k, at M_QHDR + 8 k; written by the producer with the request's first tile.
// M_F0, M_F0 + 1: the merge generation of the head / tail sequence, read before arriving.
// M_VCTA: the CTA's place in the schedule (its partial slots and share of a merge).
enum : int {
  M_ABORT = 0, M_LAST = 1, M_WCNT = 3, M_WSUM = 4, M_HEAD = 16, M_TAIL = 24, M_TMEM = 30,
  M_ZERO = 32, M_QHDR = 40, M_F0 = 56, M_VCTA = 58
};
constexpr int kMiscBytes = 256;

// ------------------------------------------------------------------ per-request geometry

struct ReqInfo {
  int32_t L, qlen, row0, tiles;
};

// Rows, context and tile count of request r, from cu_seqlens_q (never a division of a
// flat row index: ROCm/ATOM PR 2122, section 2) and context_lens.  Bad data gives 0
// tiles and a PA_DEV_* flag.
__device__ __forceinline__ ReqInfo request_info(const KParams &p, int r, uint32_t &fl) {
  ReqInfo ri;
  ri.L = p.context_lens[r];
  if (p.q_uniform > 0) {
    ri.qlen = p.q_uniform;
    ri.row0 = r * p.q_uniform;
    if (p.cu_q != nullptr && (p.cu_q[r] != ri.row0 || p.cu_q[r + 1] != ri.row0 + ri.qlen))
      fl |= PA_DEV_NOT_UNIFORM;
  } else {
    ri.row0 = p.cu_q[r];
    ri.qlen = p.cu_q[r + 1] - ri.row0;
  }
  ri.tiles = 0;
  if (ri.qlen < 0 || ri.qlen > p.max_q || ri.row0 < 0 || ri.row0 + ri.qlen > p.num_rows) {
    fl |= PA_DEV_BAD_QLEN;
    ri.qlen = 0;
    return ri;
  }
  if (ri.L < 0 || ri.L > p.max_ctx || ((ri.L + p.ps - 1) >> p.ps_shift) > p.bt_stride) {
    fl |= PA_DEV_BAD_CONTEXT;
    return ri;
  }
  if (ri.qlen == 0) return ri;
  if (ri.L < ri.qlen) fl |= PA_DEV_BAD_QLEN;
  if (p.sparse) {
    int ns = p.nsel[r];
    if (ns < 0 || ns > p.sel_stride) {
      fl |= PA_DEV_BAD_SELECTED;
      ns = ns < 0 ? 0 : p.sel_stride;
    }
    ri.tiles = (ns + p.ppt - 1) / p.ppt;
  } else {
    ri.tiles = (ri.L + kTile - 1) / kTile;
  }
  return ri;
}

// Sequence-aligned schedule: place c (< cst[B]) is chunk j of the k CTAs of sequence
// (r, h), whose nt tiles start at global tile gs.
__device__ __forceinline__ void aligned_seq(const KParams &p, const int32_t *tstart, int c, int &r,
                                            int &h, int &j, int &k, int &nt, int &gs) {
  const int B = p.num_seqs;
  const int32_t *cst = tstart + B + 2;
  int lo = 0, hi = B - 1;  // first r with cst[r + 1] > c
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (cst[mid + 1] > c)
      hi = mid;
    else
      lo = mid + 1;
  }
  r = lo;
  k = (cst[r + 1] - cst[r]) / p.Hkv;
  const int loc = c - cst[r];
  h = loc / k;
  j = loc - h * k;
  nt = tstart[r + 1] - tstart[r];
  gs = tstart[r] * p.Hkv + h * nt;
}

// The tile range [a, b) of schedule place c.
__device__ __forceinline__ void cta_range(const KParams &p, const int32_t *tstart, int c, int &a,
                                       int &b) {
  const int B = p.num_seqs, T = tstart[B] * p.Hkv;
  if (!p.sched_partition) {
    const int32_t *cst = tstart + B + 2;
    if (cst[B + 1]) {  // sequence-aligned: chunk j of the k CTAs of sequence (r, h)
      a = b = T;
      if (c >= cst[B]) return;
      int r, h, j, k, nt, gs;
      aligned_seq(p, tstart, c, r, h, j, k, nt, gs);
      const int s_last = cst[B + 1] >> 1;
      if (s_last > 0 && h == p.Hkv - 1 && cst[r + 1] == cst[B]) {
        // the grid's last sequence: its last CTA takes s_last tiles, the others share the rest
        const int rest = nt - s_last;
        a = gs + (j < k - 1 ? j * rest / (k - 1) : rest);
        b = gs + (j < k - 1 ? (j + 1) * rest / (k - 1) : nt);
        return;
      }
      a = gs + j * nt / k;
      b = gs + (j + 1) * nt / k;
      return;
    }
    const int C = (T + p.grid - 1) / p.grid;
    a = min(T, c * C);
    b = min(T, a + C);
    return;
  }
  const int s = c / p.maxch, k = c - s * p.maxch;
  const int r = s / p.Hkv, h = s - r * p.Hkv;
  a = b = 0;
  if (r >= B) return;
  const int nt = tstart[r + 1] - tstart[r];
  const int gs = tstart[r] * p.Hkv + h * nt, ge = gs + nt;
  a = min(ge, gs + k * p.part_tiles);
  b = min(ge, a + p.part_tiles);
}

// Exclusive prefix of tile counts over requests into tstart[0..B] (shared memory).
// Returns this thread's PA_DEV_* flags (reported once the kernel may write) and leaves
// the CTA's tile range [a, b) in wsum[0], wsum[1].
//
// Then the CTA schedule (balanced mode).  When there are no more sequences (request, KV
// head) than CTAs, every sequence may get a whole number of CTAs: the smallest budget X of
// work per CTA (tiles x query tokens) with sum_r ceil(nt_r q_r / X) <= floor(grid / Hkv)
// is found by bisection, and sequence r gets k_r = min(nt_r, ceil(nt_r q_r / X)) CTAs of
// equal shares.  No CTA then holds the end of one sequence and the start of another, which
// would stop all of its warps for a merge in mid-stream.  This is taken when X is no
// larger than (C + 2) q_max, C = ceil(T / grid) tiles being the equal chunk of the other
// mode.  cstart = tstart + B + 2 holds the exclusive prefix of k_r * Hkv; cstart[B + 1] =
// 1 + 2 s marks this mode, s > 0 being the share of the grid's last CTA when no CTA is
// left over.  Otherwise (cstart[B + 1] = 0) CTAs take equal chunks of C tiles.
// (Not inlined: it runs once, and its temporaries must not crowd the loops' registers.)
__device__ __noinline__ uint32_t scan_tiles(const KParams &p, int32_t *tstart, int32_t *wsum) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int NW = kThreads / 32;
  const int B = p.num_seqs;
  const int per = (B + kThreads - 1) / kThreads;
  const int r0 = min(B, tid * per), r1 = min(B, r0 + per);
  int32_t *cst = tstart + B + 2;
  uint32_t fl = 0;
  int local = 0;
  for (int r = r0; r < r1; ++r) {
    const ReqInfo ri = request_info(p, r, fl);
    tstart[r] = ri.tiles;
    cst[r] = ri.tiles * max(ri.qlen, 1);  // work of one head of the request (until replaced)
    local += ri.tiles;
  }
  int inc = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += v;
  }
  if (lane == 31) wsum[warp] = inc;
  __syncthreads();
  if (tid == 0) {
    int run = 0;
    for (int w = 0; w < NW; ++w) {
      const int v = wsum[w];
      wsum[w] = run;
      run += v;
    }
    tstart[B] = run;
  }
  __syncthreads();
  int run = wsum[warp] + inc - local;
  for (int r = r0; r < r1; ++r) {
    const int n = tstart[r];
    tstart[r] = run;
    run += n;
  }
  __syncthreads();
  if (warp == 0) {  // the schedule: one warp, no further block barriers
    const uint32_t full = 0xffffffffu;
    uint32_t ne = 0, wm = 0, qm = 1;
    unsigned long long wt = 0;
    for (int r = lane; r < B; r += 32) {
      const int nt = tstart[r + 1] - tstart[r];
      ne += nt > 0;
      wt += (uint32_t)cst[r];
      wm = max(wm, (uint32_t)cst[r]);
      if (nt > 0) qm = max(qm, (uint32_t)(cst[r] / nt));
    }
    ne = __reduce_add_sync(full, ne);
    wm = __reduce_max_sync(full, wm);
    qm = __reduce_max_sync(full, qm);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) wt += __shfl_xor_sync(full, wt, o);
    const uint32_t G = (uint32_t)(p.grid / p.Hkv);
    bool aligned = !p.sched_partition && tstart[B] > 0 && ne <= G;
    uint32_t lo = 1;
    if (aligned) {
      // lower bound: the average work per CTA; upper bounds that are feasible: the largest
      // request (one CTA each), and W / (G - E) (sum ceil(w / X) < W / X + E <= G).
      lo = (uint32_t)((wt + G - 1) / G);
      uint32_t hi = wm;
      if (lo < 1) lo = 1;
      if (G > ne) {
        const unsigned long long b = (wt + (G - ne) - 1) / (G - ne);
        if (b < hi) hi = (uint32_t)b;
      }
      if (hi < lo) lo = hi;
      while (lo < hi) {
        const uint32_t mid = (lo + hi) >> 1;
        uint32_t cnt = 0;
        for (int r = lane; r < B; r += 32) {
          const uint32_t nt = (uint32_t)(tstart[r + 1] - tstart[r]);
          const uint32_t q = ((uint32_t)cst[r] + mid - 1) / mid;
          cnt += min(q, nt);
        }
        cnt = __reduce_add_sync(full, cnt);
        if (cnt <= G)
          hi = mid;
        else
          lo = mid + 1;
      }
      // Against equal chunks of C = ceil(T / grid) tiles, whose CTAs may straddle two
      // sequences (a merge in mid-stream, some two tile-times): whole sequences only while
      // their budget is no larger than such a chunk's worst case.
      const uint32_t T = (uint32_t)tstart[B] * (uint32_t)p.Hkv;
      const uint32_t C = (T + (uint32_t)p.grid - 1) / (uint32_t)p.grid;
      aligned = lo <= (C + 2) * qm;
    }
    if (aligned) {
      // k_r at that budget (cst[r] turns from work into k_r, lane by lane), and the last
      // request that has CTAs.
      uint32_t tot = 0;
      int r_last = -1, q_last = 1;
      for (int c0 = 0; c0 < B; c0 += 32) {
        const int r = c0 + lane;
        int k = 0, nt = 0, w = 0;
        if (r < B) {
          nt = tstart[r + 1] - tstart[r];
          w = cst[r];
          k = (int)min(((uint32_t)w + lo - 1) / lo, (uint32_t)nt);
          cst[r] = k;
        }
        tot += (uint32_t)k;
        const unsigned used = __ballot_sync(full, k > 0);
        if (used) {
          const int top = 31 - __clz(used);
          q_last = __shfl_sync(full, nt > 0 ? w / nt : 1, top);
          r_last = c0 + top;
        }
      }
      tot = __reduce_add_sync(full, tot);
      __syncwarp();
      // With no CTA left over, the last CTA of the grid starts last (after the previous
      // launch's final merge and its own prologue, some 6 tile-times at one query token):
      // it takes fewer tiles.  (CTAs left over sit at the end of the grid and take those
      // late SMs themselves.)
      int s_last = 0;
      if (tot == G && r_last >= 0) {
        const int nt = tstart[r_last + 1] - tstart[r_last], k = cst[r_last];
        const int q = max(q_last, 1), pt = max(1, (6 + q / 2) / q);
        if (k >= 2) s_last = max(1, nt / k - pt);
      }
      int carry = 0;
      for (int c0 = 0; c0 < B; c0 += 32) {
        const int r = c0 + lane;
        const int k = r < B ? cst[r] * p.Hkv : 0;
        int kin = k;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int v = __shfl_up_sync(full, kin, o);
          if (lane >= o) kin += v;
        }
        if (r < B) cst[r] = carry + kin - k;
        carry += __shfl_sync(full, kin, 31);
      }
      if (lane == 0) {
        cst[B] = carry;
        cst[B + 1] = 1 + 2 * s_last;
      }
    } else if (lane == 0) {
      cst[B + 1] = 0;
    }
    __syncwarp();
    if (lane == 0) {  // this CTA's range, for every thread (wsum is free by now)
      int a, b;
      const int v = blockIdx.x;
      cta_range(p, tstart, v, a, b);
      wsum[0] = a;
      wsum[1] = b;
      wsum[M_VCTA - M_WSUM] = v;
    }
  }
  __syncthreads();
  return fl;
}

// Global tile index -> (request, KV head, tile within the request's head).
__device__ __forceinline__ void locate(const int32_t *tstart, int B, int Hkv, int gt, int &r,
                                       int &h, int &tile) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {  // first r with tstart[r + 1] * Hkv > gt
    const int mid = (lo + hi) >> 1;
    if (tstart[mid + 1] * Hkv > gt)
      hi = mid;
    else
      lo = mid + 1;
  }
  r = lo;
  const int nt = tstart[r + 1] - tstart[r];
  const int off = gt - tstart[r] * Hkv;
  h = off / nt;
  tile = off - h * nt;
}

// CTAs that hold partials of sequence (r, h) whose tiles are [gs, ge).
__device__ __forceinline__ void seq_ctas(const KParams &p, const int32_t *tstart, int r, int h,
                                         int gs, int ge, int &c_first, int &n) {
  if (!p.sched_partition) {
    const int32_t *cst = tstart + p.num_seqs + 2;
    if (cst[p.num_seqs + 1]) {
      const int k = (cst[r + 1] - cst[r]) / p.Hkv;
      c_first = cst[r] + h * k;
      n = k;
      return;
    }
    const int T = tstart[p.num_seqs] * p.Hkv;
    const int C = (T + p.grid - 1) / p.grid;
    c_first = gs / C;
    n = (ge - 1) / C - c_first + 1;
  } else {
    c_first = (r * p.Hkv + h) * p.maxch;
    n = (ge - gs + p.part_tiles - 1) / p.part_tiles;
  }
}

// Partial slot of CTA c for a sequence: the CTA where the sequence starts writes its
// "tail" slot 2c + 1; every later CTA writes its "head" slot 2c.
__device__ __forceinline__ int slot_of(int c, int c_first) { return c == c_first ? 2 * c + 1 : 2 * c; }

// --------------------------------------------------------------------- shared-memory map

// Shared-memory map: every address is computed once at kernel entry and kept in
// registers (no reads of the parameter block inside the loops).
struct Smem {
  uint8_t *base;           // generic pointer to the 1024-aligned base
  uint32_t sb;             // its shared-window address
  uint32_t stage_bytes, nstage, q0, qslot_bytes, merge_a, merge_ml, bar0;
  int32_t *tstart_p, *misc_p;
  StageMeta *meta_p;
  __device__ static Smem make(uint8_t *b, const KParams &p) {
    Smem m;
    m.base = b;
    m.sb = smem_u32(b);
    m.stage_bytes = p.stage_bytes;
    m.nstage = p.nstage;
    m.q0 = m.sb + p.off_q;
    m.qslot_bytes = p.qslot_bytes;
    m.merge_a = m.sb + p.off_merge;
    m.merge_ml = m.merge_a + p.xslots * 8192;
    m.bar0 = m.sb + p.off_bar;
    m.tstart_p = reinterpret_cast<int32_t *>(b + p.off_tstart);
    m.misc_p = reinterpret_cast<int32_t *>(b + p.off_misc);
    m.meta_p = reinterpret_cast<StageMeta *>(b + p.off_meta);
    return m;
  }
  __device__ uint32_t stage(int s) const { return sb + s * stage_bytes; }
  __device__ uint32_t qslot(int k) const { return q0 + k * qslot_bytes; }
  __device__ uint32_t merge() const { return merge_a; }
  __device__ uint32_t merge_ml_at(int k) const { return merge_ml + k * 512; }
  __device__ int32_t *tstart() const { return tstart_p; }
  __device__ StageMeta *meta(int s) const { return meta_p + s; }
  __device__ uint32_t full(int s) const { return bar0 + 8 * s; }
  __device__ uint32_t empty(int s) const { return bar0 + 8 * (nstage + s); }
  __device__ uint32_t qempty(int k) const { return bar0 + 8 * (2 * nstage + k); }
  __device__ uint32_t consbar() const { return bar0 + 8 * (2 * nstage + 2); }
  __device__ int32_t *misc() const { return misc_p; }
};


// Waits for stage s to hold CTA tile gt (fill parity `parity`).  A consumer that skipped
// the stage's previous tile may find that fill not yet landed, which the parity alone
// cannot tell from this one: the tile id the producer wrote decides.
__device__ __forceinline__ bool wait_tile(const Smem &sm, int s, uint32_t parity, int gt) {
  const volatile int32_t *id = &sm.meta(s)->gtile;
  if (mbar_try_wait(sm.full(s), parity) && *id == gt) return true;
  const long long t0 = clock64();
  while (!(mbar_try_wait(sm.full(s), parity) && *id == gt)) {
    if (clock64() - t0 > kWaitCycles) return false;
  }
  return true;
}

// Counts this CTA's partial of split sequence `seq` (nc CTAs): one thread, after the
// partial's stores are fenced.  f0 is the sequence's merge generation, read by this CTA
// before it arrives (no arrival of this call can bump it before every CTA has).  The
// last CTA to arrive resets the arrival counter (all have arrived) and bumps the
// generation, which releases the CTAs that wait for it.  misc[M_LAST + k] says whether this
// CTA was the last (k: 0 head, 1 tail).
__device__ __forceinline__ void arrive_split(const KParams &p, const Smem &sm, int seq, int nc,
                                             int f0, int k) {
  const int old = atomicAdd(p.counters + seq, 1);
  const bool last = old == nc - 1;
  if (last) {
    __threadfence();  // the other CTAs' partials (fenced before their arrivals) are visible
    *reinterpret_cast<volatile int32_t *>(p.counters + seq) = 0;
    *reinterpret_cast<volatile int32_t *>(p.flags + seq) = f0 + 1;
  }
  sm.misc()[M_LAST + k] = last ? 1 : 0;
}

// Waits (bounded) until the merge generation at `flag` differs from f0.  False on timeout.
__device__ __forceinline__ bool wait_flag(const int32_t *flag, int f0) {
  const volatile int32_t *v = flag;
  if (*v != f0) return true;
  const long long t0 = clock64();
  while (*v == f0) {
    if (clock64() - t0 > kWaitCycles) return false;
    __nanosleep(64);
  }
  return true;
}

// Shared-window address of the zero line.
__device__ __forceinline__ uint32_t zero_line(const Smem &sm) { return smem_u32(sm.misc() + M_ZERO); }

__device__ __forceinline__ void raise_flag(const KParams &p, const Smem &sm, uint32_t f) {
  atomicOr(p.status, f);
  if (f & PA_DEV_TIMEOUT) atomicExch(&sm.misc()[M_ABORT], 1);
}

}  // namespace pa
