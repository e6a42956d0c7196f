// sv_kernel.cuh -- the persistent verification kernel, generic over the
// problem (chain or tree).  A problem type P provides:
//   int n_req, ipr, chunk_el, es, V; bool bulk; Ws ws;
//   void preamble(Shared&, PosTables&, int4* scan_tmp) const
//        -> fills the position tables, sets sh.n_pos (all threads call it)
//   const char* row_ptr(const PosTables&, int pos, int row_local, int& kind,
//                       Scale2& c) const
//   void finalize(Shared&, const PosTables&, int pos, int ctid) const
//        (called by the kConsumers consumer threads)
#pragma once

#include "sv_rowpass.cuh"

namespace sv {

// Position of the request that owns flat row `row`: the largest pos with
// rstart[pos] <= row, searched forward from a hint (claims of one CTA are
// increasing).
__device__ __forceinline__ int find_pos(const int* rstart, int n_pos, int row, int hint) {
  int p = hint;
  if (p < 0 || p >= n_pos || rstart[p] > row) {
    int lo = 0, hi = n_pos - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (rstart[mid] <= row) lo = mid;
      else hi = mid - 1;
    }
    return lo;
  }
  while (p + 1 < n_pos && rstart[p + 1] <= row) ++p;
  return p;
}

template <class P>
__device__ void producer_loop(const P& prob, Shared& sh, const PosTables& tab,
                              unsigned char* stages) {
  const int n_pos = sh.n_pos;
  const int n_rows = tab.rstart[n_pos];
  const unsigned n_items = static_cast<unsigned>(n_rows) * static_cast<unsigned>(prob.ipr);
  unsigned item = atomicAdd(&prob.ws.hdr->work_counter, 1u);
  int hint = 0;
  for (int it = 0;; ++it) {
    const int stage = it % kStages;
    const bool have = item < n_items;
    const unsigned next = have ? atomicAdd(&prob.ws.hdr->work_counter, 1u) : 0u;
    if (it >= kStages) {
      const uint64_t lim = sh.timed_out ? kWaitLimitAfterTimeoutNs : kWaitLimitNs;
      if (!mbar_wait_bounded(&sh.empty[stage], ((it / kStages) - 1) & 1, lim)) {
        sh.timed_out = 1;
        record_error(&prob.ws.hdr->error, 0x10);
      }
    }
    StageMeta& mt = sh.meta[stage];
    if (!have) {
      mt.item = -1;
      mbar_arrive(&sh.full[stage]);
      break;
    }
    const int row = static_cast<int>(item / prob.ipr);
    const int chunk = static_cast<int>(item % prob.ipr);
    const int pos = find_pos(tab.rstart, n_pos, row, hint);
    hint = pos;
    int kind;
    Scale2 c;
    const char* rp = prob.row_ptr(tab, pos, row - tab.rstart[pos], kind, c);
    const int el_base = chunk * prob.chunk_el;
    const int n_el = min(prob.chunk_el, prob.V - el_base);
    mt.item = static_cast<int>(item);
    mt.pos = pos;
    mt.row = row;
    mt.kind = kind;
    mt.n_el = n_el;
    mt.el_base = el_base;
    mt.c_hi = c.hi;
    mt.c_lo = c.lo;
    mt.src = rp + static_cast<size_t>(el_base) * prob.es;
    if (prob.bulk) {
      const uint32_t bytes = static_cast<uint32_t>(n_el * prob.es);
      mbar_arrive_expect_tx(&sh.full[stage], bytes);
      bulk_copy_g2s(stages + static_cast<size_t>(stage) * kChunkBytes, mt.src, bytes,
                    &sh.full[stage]);
    } else {
      mbar_arrive(&sh.full[stage]);
    }
    item = next;
  }
}

template <class P>
__device__ void consumer_loop(const P& prob, Shared& sh, const PosTables& tab,
                              unsigned char* stages) {
  const int ctid = threadIdx.x;  // 0 .. kConsumers-1
  const int warp = ctid >> 5, lane = ctid & 31;
  for (int j = 0;; ++j) {
    const int stage = j % kStages;
    const uint64_t lim = sh.timed_out ? kWaitLimitAfterTimeoutNs : kWaitLimitNs;
    if (!mbar_wait_bounded(&sh.full[stage], (j / kStages) & 1, lim)) {
      sh.timed_out = 1;
      record_error(&prob.ws.hdr->error, 0x10);
    }
    const StageMeta mt = sh.meta[stage];
    if (mt.item < 0) break;
    const unsigned char* sp = stages + static_cast<size_t>(stage) * kChunkBytes;
    MS ms{kNegInf, 0.f};
    VI vi{kNegInf, 0x7fffffff};
    const bool fast = prob.bulk && prob.es == 2;
    if (mt.kind == KIND_ARGMAX) {
      if (fast)
        reduce_chunk_bf16<KIND_ARGMAX>(mt, reinterpret_cast<const uint4*>(sp), &sh.empty[stage],
                                       ctid, lane, ms, vi);
      else
        reduce_chunk_generic<KIND_ARGMAX>(mt, reinterpret_cast<const char*>(sp), prob.bulk,
                                          prob.es, &sh.empty[stage], ctid, lane, ms, vi);
      vi = warp_reduce_vi(vi);
      if (lane == 0) sh.red_vi[j & 1][warp] = vi;
    } else {
      if (fast)
        reduce_chunk_bf16<KIND_SOFTMAX>(mt, reinterpret_cast<const uint4*>(sp),
                                        &sh.empty[stage], ctid, lane, ms, vi);
      else
        reduce_chunk_generic<KIND_SOFTMAX>(mt, reinterpret_cast<const char*>(sp), prob.bulk,
                                           prob.es, &sh.empty[stage], ctid, lane, ms, vi);
      ms = warp_reduce_ms(ms, Scale2{mt.c_hi, mt.c_lo});
      if (lane == 0) sh.red_ms[j & 1][warp] = ms;
    }
    named_sync(1, kConsumers);
    // a finalize flagged during the previous iteration runs now
    const int fin = sh.fin_pending;
    if (fin >= 0) {
      prob.finalize(sh, tab, fin, ctid);
      if (ctid == 0) sh.fin_pending = -1;
      named_sync(1, kConsumers);
    }
    if (ctid == 0) {
      float2 part;
      if (mt.kind == KIND_ARGMAX) {
        VI r = sh.red_vi[j & 1][0];
        for (int w = 1; w < kConsumerWarps; ++w) r = vi_better(r, sh.red_vi[j & 1][w]);
        part = make_float2(r.v, __int_as_float(r.i));
      } else {
        MS r = sh.red_ms[j & 1][0];
        const Scale2 c{mt.c_hi, mt.c_lo};
        for (int w = 1; w < kConsumerWarps; ++w) r = ms_combine(r, sh.red_ms[j & 1][w], c);
        part = make_float2(r.m, r.s);
      }
      prob.ws.partials[static_cast<size_t>(mt.row) * prob.ipr + (mt.el_base / prob.chunk_el)] =
          part;
      __threadfence();
      const int rows = tab.rstart[mt.pos + 1] - tab.rstart[mt.pos];
      const unsigned need = static_cast<unsigned>(rows * prob.ipr);
      const int b = info_req(tab.info[mt.pos]);
      const unsigned old = atomicAdd(&prob.ws.tickets[b], 1u);
      if (old + 1u == need) {
        __threadfence();
        sh.fin_pending = mt.pos;
      }
    }
  }
  named_sync(1, kConsumers);
  const int fin = sh.fin_pending;
  if (fin >= 0) {
    prob.finalize(sh, tab, fin, ctid);
    if (ctid == 0) sh.fin_pending = -1;
  }
}

template <class P>
__global__ void __launch_bounds__(kThreads, 1) verify_kernel(const P prob) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* stages = smem_raw;
  Shared& sh = *reinterpret_cast<Shared*>(smem_raw + kStages * kChunkBytes);
  unsigned char* tail = smem_raw + kStages * kChunkBytes + ((sizeof(Shared) + 15) & ~size_t(15));
  PosTables tab;
  tab.scale = reinterpret_cast<float2*>(tail);
  tab.aux = reinterpret_cast<unsigned long long*>(tail + sizeof(float2) * prob.n_req);
  tab.info = reinterpret_cast<int*>(tail + (sizeof(float2) + (P::kAux ? 8 : 0)) * prob.n_req);
  tab.rstart = tab.info + prob.n_req;
  __shared__ int4 scan_tmp[kThreads / 32];

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sh.full[s], 1);
      mbar_init(&sh.empty[s], kConsumerWarps);
    }
    fence_mbar_init();
    sh.fin_pending = -1;
    sh.timed_out = 0;
  }
  prob.preamble(sh, tab, scan_tmp);
  __syncthreads();

  if (threadIdx.x >= kConsumers) {
    if (threadIdx.x == kConsumers) producer_loop(prob, sh, tab, stages);
  } else {
    consumer_loop(prob, sh, tab, stages);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned d = atomicAdd(&prob.ws.hdr->done_ctas, 1u);
    if (d + 1u == gridDim.x) {
      prob.ws.hdr->work_counter = 0u;
      prob.ws.hdr->done_ctas = 0u;
      __threadfence();
    }
  }
}

}  // namespace sv
