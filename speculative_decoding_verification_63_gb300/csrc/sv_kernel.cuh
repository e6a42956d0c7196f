// sv_kernel.cuh -- the persistent verification kernel, generic over the
// problem (chain or tree).
//
// One CTA per SM, four warp roles:
//   warps 0..15  consumers: each warp reduces its sixteenth of every staged
//                chunk, releases the stage as soon as the data is in
//                registers, and posts its partial into the result ring.
//   warp  16     producer: claims chunks with a global atomic counter and
//                moves them into the 4-stage ring with 1-D bulk copies.
//   warp  17     bookkeeper: takes result slots in order, combines the 16
//                per-warp partials of a chunk (max first, one rescale, a
//                sum), stores one partial per chunk and bumps the per-request
//                tickets in lane-parallel batches; a request whose last
//                chunk is in joins the finalize list.
//   warps 18..21 finalizer group: runs each listed request's finalize while
//                the consumers keep streaming.
// Every hand-off is an mbarrier (or, for the finalize list, a counter polled
// with back-off); all waits are bounded.
//
// A problem type P provides:
//   int n_req, ipr, chunk_el, es, V; bool bulk; Ws ws;
//   static constexpr int kAuxBytes  (per-position aux table, 0, 8 or 16)
//   void preamble(Shared&, PosTables&, int4* scan_tmp) const  (all threads)
//   void fill_stage(const PosTables&, int row_local, StageMeta&) const
//        -> kind, scale, source pointer(s) and aux of a chunk (producer)
//   float2 consume(const StageMeta&, const unsigned char* stage,
//                  uint64_t* empty_bar, int ctid, int lane) const
//        -> the warp's partial of a chunk; arrives on empty_bar once the
//           staged data is no longer needed (consumer warps)
//   void finalize(Shared&, const PosTables&, int pos, int ftid) const
//        (called by the kFinThreads finalizer threads)
//   void last_cta_reset() const   (the last CTA to finish, after every other)
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

__device__ __forceinline__ uint64_t wait_limit(const Shared& sh) {
  return sh.timed_out ? kWaitLimitAfterTimeoutNs : kWaitLimitNs;
}

__device__ __forceinline__ void wait_or_flag(Shared& sh, uint64_t* bar, uint32_t parity,
                                             int* err) {
  if (!mbar_wait_bounded(bar, parity, wait_limit(sh))) {
    sh.timed_out = 1;
    record_error(err, 0x10);
  }
}

template <class P>
__device__ void producer_loop(const P& prob, Shared& sh, const PosTables& tab,
                              unsigned char* stages) {
  int* err = &prob.ws.hdr->error;
  const int n_pos = sh.n_pos;
  const int n_rows = tab.rstart[n_pos];
  const unsigned n_items = static_cast<unsigned>(n_rows) * static_cast<unsigned>(prob.ipr);
  unsigned item = atomicAdd(&prob.ws.hdr->work_counter, 1u);
  int hint = 0;
  for (int it = 0;; ++it) {
    const int stage = it % kStages;
    const int rs = it % kResSlots;
    const bool have = item < n_items;
    const unsigned next = have ? atomicAdd(&prob.ws.hdr->work_counter, 1u) : 0u;
    if (it >= kStages) wait_or_flag(sh, &sh.empty[stage], ((it / kStages) - 1) & 1, err);
    if (it >= kResSlots) wait_or_flag(sh, &sh.res_free[rs], ((it / kResSlots) - 1) & 1, err);
    StageMeta& mt = sh.meta[stage];
    ResMeta& rm = sh.res_meta[rs];
    if (!have) {
      mt.item = -1;
      rm.item = -1;
      mbar_arrive(&sh.res_done[rs]);
      mbar_arrive(&sh.full[stage]);
      break;
    }
    const int row = static_cast<int>(item / prob.ipr);
    const int chunk = static_cast<int>(item % prob.ipr);
    const int pos = find_pos(tab.rstart, n_pos, row, hint);
    hint = pos;
    mt.item = static_cast<int>(item);
    mt.pos = pos;
    mt.row = row;
    mt.el_base = chunk * prob.chunk_el;
    mt.n_el = min(prob.chunk_el, prob.V - mt.el_base);
    mt.src2 = nullptr;
    prob.fill_stage(tab, row - tab.rstart[pos], mt);
    rm.item = static_cast<int>(item);
    rm.pos = pos;
    rm.slot = row * prob.ipr + chunk;
    rm.kind = mt.kind;
    rm.c_hi = mt.c_hi;
    rm.c_lo = mt.c_lo;
    mbar_arrive(&sh.res_done[rs]);
    if (prob.bulk) {
      // one or two row pieces of n_el elements: [0, half) and [half, 2 half)
      const uint32_t bytes = static_cast<uint32_t>(mt.n_el * prob.es);
      unsigned char* dst = stages + static_cast<size_t>(stage) * kChunkBytes;
      mbar_arrive_expect_tx(&sh.full[stage], mt.src2 ? 2u * bytes : bytes);
      bulk_copy_g2s(dst, mt.src, bytes, &sh.full[stage]);
      if (mt.src2) bulk_copy_g2s(dst + kChunkBytes / 2, mt.src2, bytes, &sh.full[stage]);
    } else {
      mbar_arrive(&sh.full[stage]);
    }
    item = next;
  }
}

template <class P>
__device__ void consumer_loop(const P& prob, Shared& sh, unsigned char* stages) {
  int* err = &prob.ws.hdr->error;
  const int ctid = threadIdx.x;  // 0 .. kConsumers-1
  const int warp = ctid >> 5, lane = ctid & 31;
  for (int j = 0;; ++j) {
    const int stage = j % kStages;
    const int rs = j % kResSlots;
    wait_or_flag(sh, &sh.full[stage], (j / kStages) & 1, err);
    const StageMeta mt = sh.meta[stage];
    if (mt.item < 0) {
      if (lane == 0) mbar_arrive(&sh.res_done[rs]);
      break;
    }
    const unsigned char* sp = stages + static_cast<size_t>(stage) * kChunkBytes;
    const float2 part = prob.consume(mt, sp, &sh.empty[stage], ctid, lane);
    if (lane == 0) {
      sh.res_part[rs][warp] = part;
      mbar_arrive(&sh.res_done[rs]);  // release: the partial is visible to the bookkeeper
    }
  }
}

// Bookkeeper: book the collected chunks (lane i holds chunk i < nb) and
// publish completed requests to the finalize list.
template <class P>
__device__ void bk_flush(const P& prob, Shared& sh, const PosTables& tab, int lane, int nb,
                         int e_pos) {
  if (nb == 0) return;
  __threadfence();  // the partials -> GPU scope before the tickets
  bool done = false;
  if (lane < nb) {
    const int rows = tab.rstart[e_pos + 1] - tab.rstart[e_pos];
    const unsigned need = static_cast<unsigned>(rows * prob.ipr);
    const unsigned old = atomic_add_acq_rel(&prob.ws.tickets[info_req(tab.info[e_pos])], 1u);
    done = old + 1u == need;
  }
  const unsigned dmask = __ballot_sync(0xffffffffu, done);
  if (dmask) {
    __threadfence();  // every partial of the completed requests is visible
    const unsigned tail = sh.fin_tail;
    // room: the finalizer consumes in order; wait (bounded) if the list is full
    const unsigned need_room = tail + __popc(dmask);
    volatile unsigned* vhead = &sh.fin_head;
    if (need_room - *vhead > static_cast<unsigned>(kFinCap)) {
      const uint64_t t0 = globaltimer_ns();
      while (need_room - *vhead > static_cast<unsigned>(kFinCap)) {
        __nanosleep(200);
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
          if (lane == 0) record_error(&prob.ws.hdr->error, 0x10);
          break;
        }
      }
    }
    if (done)
      reinterpret_cast<volatile int*>(sh.fin_q)[(tail + __popc(dmask & ((1u << lane) - 1u))) %
                                                 kFinCap] = e_pos;
    __syncwarp();
    if (lane == 0) {
      __threadfence_block();
      *reinterpret_cast<volatile unsigned*>(&sh.fin_tail) = need_room;
    }
  }
  __syncwarp();
}

// Bookkeeper warp: per chunk, copy the consumer warps' partials to the
// workspace (one coalesced 128-byte store; the finalize merges them), then
// book the chunk's ticket in lane-parallel batches.
template <class P>
__device__ void bookkeeper_loop(const P& prob, Shared& sh, const PosTables& tab) {
  int* err = &prob.ws.hdr->error;
  const int lane = threadIdx.x & 31;
  int nb = 0;  // chunks collected, not yet booked
  int e_pos = 0;
  for (int j = 0;; ++j) {
    const int rs = j % kResSlots;
    const uint32_t par = (j / kResSlots) & 1;
    if (nb > 0 && !mbar_test_wait(&sh.res_done[rs], par)) {
      bk_flush(prob, sh, tab, lane, nb, e_pos);
      nb = 0;
    }
    wait_or_flag(sh, &sh.res_done[rs], par, err);
    const ResMeta rm = sh.res_meta[rs];
    if (rm.item < 0) break;
    // combine the consumer warps' partials of the chunk (lanes 0..15)
    const float2 p = lane < kConsumerWarps ? sh.res_part[rs][lane] : make_float2(kNegInf, 0.f);
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh.res_free[rs]);
    float2 tot;
    if (rm.kind == KIND_ARGMAX) {
      const VI v = warp_reduce_vi(VI{p.x, lane < kConsumerWarps ? __float_as_int(p.y)
                                                                : 0x7fffffff});
      tot = make_float2(v.v, __int_as_float(v.i));
    } else if (rm.kind == KIND_RESID_PASS) {
      // residual pass: the partials are segment sums, kept one per warp
      tot = p;
    } else {
      const MS v = warp_reduce_ms(MS{p.x, p.y}, Scale2{rm.c_hi, rm.c_lo});
      tot = make_float2(v.m, v.s);
    }
    const int slot = rm.slot, pos = rm.pos;
    if (rm.kind == KIND_RESID_PASS) {
      if (lane < kConsumerWarps)
        prob.ws.partials[static_cast<size_t>(slot) * kConsumerWarps + lane] = tot;
    } else if (lane == 0) {
      prob.ws.partials[slot] = tot;
    }
    if (lane == nb) e_pos = pos;
    if (++nb == 32) {
      bk_flush(prob, sh, tab, lane, nb, e_pos);
      nb = 0;
    }
  }
  bk_flush(prob, sh, tab, lane, nb, e_pos);
  __syncwarp();
  if (lane == 0) {
    __threadfence_block();
    *reinterpret_cast<volatile unsigned*>(&sh.bk_done) = 1u;
  }
}

template <class P>
__device__ void finalizer_loop(const P& prob, Shared& sh, const PosTables& tab) {
  const int ftid = threadIdx.x - kFinBase;
  uint64_t idle_since = 0;
  unsigned backoff = 32;
  for (;;) {
    if (ftid == 0) {
      int cmd = -1;  // idle
      volatile unsigned* vtail = &sh.fin_tail;
      const unsigned tail = *vtail;
      if (sh.fin_head != tail) {
        __threadfence_block();
        cmd = reinterpret_cast<volatile int*>(sh.fin_q)[sh.fin_head % kFinCap];
        *reinterpret_cast<volatile unsigned*>(&sh.fin_head) = sh.fin_head + 1u;
        idle_since = 0;
        backoff = 32;
      } else if (*reinterpret_cast<volatile unsigned*>(&sh.bk_done) != 0u &&
                 *vtail == sh.fin_head) {
        cmd = -2;  // every chunk booked and every complete request finalized
      } else {
        const uint64_t now = globaltimer_ns();
        if (idle_since == 0) idle_since = now;
        if (now - idle_since > 2 * kWaitLimitNs) {
          record_error(&prob.ws.hdr->error, 0x10);
          cmd = -2;
        }
      }
      if (cmd == -1) {
        __nanosleep(backoff);
        backoff = min(backoff * 2u, 256u);
      }
      sh.fin_cmd = cmd;
    }
    named_sync(1, kFinThreads);
    const int cmd = sh.fin_cmd;
    named_sync(1, kFinThreads);
    if (cmd == -2) break;
    if (cmd >= 0) prob.finalize(sh, tab, cmd, ftid);
  }
}

template <class P>
__global__ void __launch_bounds__(kThreads, 1) verify_kernel(const P prob) {
  extern __shared__ __align__(1024) unsigned char smem_dyn[];
  // 128-byte aligned base (the launch adds 128 bytes of slack)
  unsigned char* smem_raw = smem_dyn + ((128u - (smem_u32(smem_dyn) & 127u)) & 127u);
  unsigned char* stages = smem_raw;
  Shared& sh = *reinterpret_cast<Shared*>(smem_raw + kStages * kChunkBytes);
  unsigned char* tail = smem_raw + kStages * kChunkBytes + ((sizeof(Shared) + 15) & ~size_t(15));
  // tables in decreasing alignment: aux (16- or 8-byte entries) at the
  // 16-byte aligned tail, then the float2 scales, then the int tables
  PosTables tab;
  tab.aux = reinterpret_cast<float4*>(tail);
  tab.scale = reinterpret_cast<float2*>(tail + static_cast<size_t>(P::kAuxBytes) * prob.n_req);
  tab.info = reinterpret_cast<int*>(tail + (sizeof(float2) + P::kAuxBytes) * prob.n_req);
  tab.rstart = tab.info + prob.n_req;
  __shared__ int4 scan_tmp[kThreads / 32];

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sh.full[s], 1);
      mbar_init(&sh.empty[s], kConsumerWarps);
    }
    for (int s = 0; s < kResSlots; ++s) {
      mbar_init(&sh.res_done[s], kConsumerWarps + 1);
      mbar_init(&sh.res_free[s], 1);
    }
    fence_mbar_init();
    sh.timed_out = 0;
    sh.fin_head = sh.fin_tail = 0u;
    sh.bk_done = 0u;
    sh.fin_cmd = -1;
  }
  prob.preamble(sh, tab, scan_tmp);
  __syncthreads();

  if (threadIdx.x < kConsumers) {
    consumer_loop(prob, sh, stages);
  } else if (threadIdx.x < kBkBase) {
    if (threadIdx.x == kProducerThread) producer_loop(prob, sh, tab, stages);
  } else if (threadIdx.x < kFinBase) {
    bookkeeper_loop(prob, sh, tab);
  } else {
    finalizer_loop(prob, sh, tab);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned d = atomicAdd(&prob.ws.hdr->done_ctas, 1u);
    if (d + 1u == gridDim.x) {
      prob.ws.hdr->work_counter = 0u;
      prob.ws.hdr->done_ctas = 0u;
      prob.last_cta_reset();
      __threadfence();
    }
  }
}

}  // namespace sv
