// pa_producer.cuh -- the producer warp: page gather into shared-memory stages.
#pragma once

#include "pa_kernel.cuh"

namespace pa {

// Bytes one valid page brings into a stage.
template <int KVT, int SM>
__device__ __forceinline__ uint32_t page_bytes(int ps) {
  if (KVT == PA_KV_BF16) return 4u * ps * kD;
  return 2u * ps * kD + (SM == PA_SCALE_PER_TOKEN ? 8u * ps : 0u);
}

// Walks tiles [a, b) in batches: each lane resolves one page of one tile (lanes
// ppt*j .. ppt*j + ppt - 1 serve tile j of the batch), so the dependent global loads
// of a whole batch (context length, selected-page entry, block-table entry) are in
// flight together.  Then, tile by tile: wait for the stage to be free, publish the
// tile's metadata, arm the stage's full barrier with the byte count, and issue the
// TMA copies (K and V rows with 128-byte swizzle, per-token scales, and the
// request's query rows at the first tile of a request).
template <int KVT, int SM>
__device__ void run_producer(const KParams &p, const Smem &sm, int a, int b, uint32_t report) {
  const int lane = threadIdx.x & 31;
  const int ppt = p.ppt, nb = 32 / ppt;
  const int slot = lane / ppt, kpg = lane - slot * ppt;
  const int32_t *tstart = sm.tstart();
  const int ps = p.ps;
  const uint64_t pol = l2_evict_first_policy();
  const uint32_t pbytes = page_bytes<KVT, SM>(ps);
  int i = 0, seg = 0;
  bool ok = true, waited_deps = false;

  for (int base = a; base < b && ok; base += nb) {
    const int gt = base + slot;
    int r = 0, h = 0, tile = 0, nt = 1, pos = -1, phys = -1;
    ReqInfo ri{0, 0, 0, 0};
    uint32_t fl = 0;
    if (gt < b) {
      locate(tstart, p.num_seqs, p.Hkv, gt, r, h, tile);
      nt = tstart[r + 1] - tstart[r];
      uint32_t seen = 0;  // request-level flags were reported by the prologue
      ri = request_info(p, r, seen);
      const int np = (ri.L + ps - 1) >> p.ps_shift;
      const int idx = tile * ppt + kpg;
      int lp = -1;
      if (!p.sparse) {
        lp = idx < np ? idx : -1;
      } else {
        int ns = p.nsel[r];
        ns = ns < 0 ? 0 : min(ns, p.sel_stride);
        if (idx < ns) {
          const int e = p.sel[(int64_t)r * p.sel_stride + idx];
          if (e < -1 || e >= np) fl |= PA_DEV_BAD_SELECTED;
          lp = (e >= 0 && e < np) ? e : -1;
        }
      }
      if (lp >= 0) {
        const int ph = p.block_table[(int64_t)r * p.bt_stride + lp];
        if (ph < 0 || (int64_t)ph >= p.num_pages)
          fl |= PA_DEV_BAD_PAGE;
        else {
          phys = ph;
          pos = lp * ps;
        }
      }
    }
    if (!waited_deps) {
      // Everything above read only index inputs; q, the caches, the scales and the
      // workspace wait for the kernels this launch depends on.  Before the wait, only
      // L2 prefetches of the first tiles' pages: they move nothing into this kernel (its
      // reads come after the wait, and L2 is where every write lands first), but they
      // let HBM fetch those pages while the previous kernel finishes.
      if (gt < b && slot < p.nstage && phys >= 0) {
        const int32_t rowp = (phys * p.Hkv + h) * ps;
        const uint32_t rb = (KVT == PA_KV_FP8_E4M3 ? 1u : 2u) * kD;
        prefetch_l2(p.k_cache + (int64_t)rowp * rb, ps * rb);
        prefetch_l2(p.v_cache + (int64_t)rowp * rb, ps * rb);
        if (SM == PA_SCALE_PER_TOKEN) {
          prefetch_l2(p.k_scale + rowp, ps * 4);
          prefetch_l2(p.v_scale + rowp, ps * 4);
        }
      }
      pdl_wait();
      if (lane == 0) trace(T_PRODUCER);
      waited_deps = true;
      if (report) atomicOr(p.status, report);
    }
    if (fl) atomicOr(p.status, fl);
    const unsigned valid_bits = __ballot_sync(~0u, phys >= 0);
    const int cut0 = ri.L - ri.qlen + 1;  // smallest causal cutoff of the request's rows
    const unsigned mask_bits = __ballot_sync(~0u, gt < b && (phys < 0 || pos + ps > cut0));
    const int nbat = min(nb, b - base);

    for (int j = 0; j < nbat; ++j) {
      const int src = j * ppt;
      const unsigned slot_bits = (ppt == 32 ? ~0u : ((1u << ppt) - 1u)) << src;
      const int rj = __shfl_sync(~0u, r, src), hj = __shfl_sync(~0u, h, src);
      const int tj = __shfl_sync(~0u, tile, src), ntj = __shfl_sync(~0u, nt, src);
      const int Lj = __shfl_sync(~0u, ri.L, src), qj = __shfl_sync(~0u, ri.qlen, src);
      const int row0j = __shfl_sync(~0u, ri.row0, src);
      const int gtj = base + j;
      const bool begin = (gtj == a) || (tj == 0);
      const bool end = (gtj == b - 1) || (tj == ntj - 1);
      const int seq_start = gtj - tj;
      const bool whole = seq_start >= a && seq_start + ntj <= b;
      const int flags = (begin ? F_BEGIN : 0) | (end ? F_END : 0) |
                        ((mask_bits & slot_bits) ? F_MASK : 0) | (whole ? F_WHOLE : 0);
      const int s = i % p.nstage;
      int waited = 1;
      if (lane == 0 && i >= p.nstage)
        waited = mbar_wait_bounded(sm.empty(s), ((i / p.nstage) - 1) & 1) ? 1 : 0;
      int qs = 0;
      if (begin) {
        qs = seg & 1;
        if (lane == 0 && waited && seg >= 2)
          waited = mbar_wait_bounded(sm.qempty(qs), ((seg >> 1) - 1) & 1) ? 1 : 0;
        ++seg;
      }
      waited = __shfl_sync(~0u, waited, 0);
      if (!waited) {
        if (lane == 0) raise_flag(p, sm, PA_DEV_TIMEOUT);
        ok = false;
        break;
      }
      StageMeta *mt = sm.meta(s);
      if (lane >= src && lane < src + ppt) {
        mt->page_pos[kpg] = pos;
        mt->page_phys[kpg] = phys;
      }
      if (lane == 0) {
        mt->r = rj;
        mt->h = hj;
        mt->tile = tj;
        mt->flags = flags;
        mt->L = Lj;
        mt->qlen = qj;
        mt->row0 = row0j;
        mt->nvalid = __popc(valid_bits & slot_bits);
        mt->gtile = gtj;
        mt->qslot = qs;
        if (begin) {
          int32_t *qh = sm.misc() + M_QHDR + 8 * qs;
          qh[0] = rj;
          qh[1] = hj;
          qh[2] = qj;
          qh[3] = row0j;
          qh[4] = Lj;
        }
      }
      __syncwarp();
      const uint32_t tx = __popc(valid_bits & slot_bits) * pbytes +
                          (begin ? (uint32_t)qj * kQRowBytes : 0u);
      if (lane == 0) mbar_arrive_expect_tx(sm.full(s), tx);
      __syncwarp();
      const uint32_t st = sm.stage(s), fb = sm.full(s);
      if (lane >= src && lane < src + ppt && phys >= 0) {
        const int32_t row = (phys * p.Hkv + hj) * ps;
        const uint32_t po = kpg * ps * 128;
        if (KVT == PA_KV_FP8_E4M3) {
          tma_load_2d(st + po, &p.tm_k, 0, row, fb, pol);
          tma_load_2d(st + 16384 + po, &p.tm_v, 0, row, fb, pol);
          if (SM == PA_SCALE_PER_TOKEN) {
            bulk_load_hint(st + 32768 + kpg * ps * 4, p.k_scale + row, ps * 4, fb, pol);
            bulk_load_hint(st + 33280 + kpg * ps * 4, p.v_scale + row, ps * 4, fb, pol);
          }
        } else {
          tma_load_2d(st + po, &p.tm_k, 0, row, fb, pol);
          tma_load_2d(st + 16384 + po, &p.tm_k, 64, row, fb, pol);
          tma_load_2d(st + 32768 + po, &p.tm_v, 0, row, fb, pol);
          tma_load_2d(st + 49152 + po, &p.tm_v, 64, row, fb, pol);
        }
      }
      if (begin && lane < qj) {
        const uint16_t *qsrc = p.q + ((int64_t)(row0j + lane) * (p.Hkv * kG) + hj * kG) * kD;
        bulk_load(sm.qslot(qs) + lane * kQRowBytes, qsrc, kQRowBytes, fb);
      }
      ++i;
    }
  }
  if (!ok && lane == 0) {
    // Let every copy already issued land before the CTA can exit.
    for (int k = max(0, i - p.nstage); k < i; ++k)
      mbar_wait_bounded(sm.full(k % p.nstage), (k / p.nstage) & 1);
  }
}

}  // namespace pa
