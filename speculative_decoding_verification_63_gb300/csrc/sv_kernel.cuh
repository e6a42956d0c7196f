// sv_kernel.cuh -- the persistent verification kernel, generic over the
// problem (chain or tree).
//
// One CTA per SM, warp roles (control warps first, so that the warp
// schedulers, which favour lower warp ids, serve them ahead of the
// always-ready consumers):
//   warp  0      producer: moves chunks into the 4-stage ring with 1-D bulk
//                copies: the CTA's share of the main pass (chunks
//                blockIdx.x + j G over the G streaming CTAs), and, ahead of
//                the next main-pass chunk, every draw-pass chunk the scout
//                has left in the shared mailbox.  The 32 lanes work out the
//                main-pass chunks 32 at a time, each keeping its chunk's
//                metadata in registers; each then puts its own chunk into
//                the ring (16-byte stores) and issues the bulk copy.
//                The producer reads only shared memory, so it never waits on
//                a global load.  With nothing left it ends the stream with
//                one sentinel per consumer group.
//   warp  1      bookkeeper: takes result slots in order, combines the 8
//                per-warp partials of a chunk (max first, one rescale, a
//                sum) or keeps the residual segment sums and stores them;
//                without control CTAs it also appends the chunk's ticket to
//                the booked queue.
//   warp  2      ticket warp (problems without control CTAs): takes booked
//                chunks in lane-parallel batches, fences, bumps the tickets;
//                a completed request joins the finalize list.
//   warp  6      draw scout (problems with draw passes; otherwise the
//                fourth finalizer): walks the CTA's static share of the
//                draw-pass claims, waits for each claimed draw to be
//                published, plans the chunk and leaves it in the mailbox.
//   warps 3..5   finalizers (3..6 without draw passes; problems without
//                control CTAs): take finalize-list entries (each warp on its
//                own, or the four together for problems that need a group)
//                while the consumers keep streaming.
//   warps 7..22  consumers, in two groups of eight that take alternate
//                chunks (so each group has two chunk times per chunk): each
//                warp reduces its eighth of the chunk, releases the stage as
//                soon as the data is in registers, and posts its partial
//                into the result ring.
// Every hand-off is an mbarrier or a shared counter polled with back-off;
// every wait is bounded.  The waits on other CTAs -- a finalize on its
// request's chunks, a scout on its claimed draw, a draw finalize on its
// draw's chunks -- only ever wait on CTAs that are running: the grid never
// exceeds the SM count and a CTA holds the whole of an SM, and none of the
// awaited work waits on the waiter.

// A problem type P provides:
//   int n_req, ipr, chunk_el, es, V; bool bulk; Ws ws;
//   static constexpr int kAuxBytes       per-position aux table (0, 8, 16)
//   static constexpr bool kWarpFinalize  finalizes run per warp (else group)
//   static constexpr bool kHasDraws      the problem publishes draw passes
//   void prefetch_args(int lane) const  L2 hints issued before the dependency wait
//   void preamble(Shared&, PosTables&, int4* scan_tmp, unsigned char* scratch) const
//        (all threads; scratch: the chunk ring, free until the preamble ends)
//   void fill_stage(const PosTables&, int row_local, StageMeta&, ResMeta&)
//        -> a main-pass chunk: kind, scale, source, ticket fields (producer)
//   void fill_resid(const P2Job&, int chunk, StageMeta&, ResMeta&) const
//        -> a draw-pass chunk (scout)
//   int ipr2                     chunks per draw
//   int poll_job(const PosTables&, int d, uint64_t limit, P2Job&) const
//        -> the draw at position d, polled until published (1), failed (0)
//           or the wait expired (-1)
//   void store_segsums_warp(int slot, int w, float4) const
//        -> the bookkeeper's store of consumer warp w's segment sums
//   float4 consume(const StageMeta&, const unsigned char* stage,
//                  uint64_t* empty_bar, int ctid, int lane) const
//        (ctid: thread index within the consumer group)
//   void finalize_warp(Shared&, const PosTables&, int code, int lane,
//                      WarpFin&) const     (kWarpFinalize)
//   void finalize(Shared&, const PosTables&, int code, int ftid) const
//                                          (!kWarpFinalize, all 4 warps)
//   static constexpr bool kHasDirectFin  some requests need no main-pass rows
//   bool direct_fin(const PosTables&, int pos) const
//        -> request at pos goes straight to the finalize list (kHasDirectFin)
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

__device__ __forceinline__ unsigned vload(const unsigned& x) {
  return *reinterpret_cast<const volatile unsigned*>(&x);
}

// Give up a bounded wait: flag the timeout (later waits of this CTA are short).
__device__ __forceinline__ void flag_timeout(Shared& sh, int* err) {
  sh.timed_out = 1;
  record_error(err, 0x10);
}

// Control CTAs (problems with kCtrl): the last n_ctrl CTAs of the grid
// stream nothing; the main pass is spread over the others.
template <class P>
__device__ __forceinline__ unsigned n_ctrl_of(const P& prob) {
  if constexpr (P::kCtrl) return static_cast<unsigned>(prob.n_ctrl);
  else return 0u;
}

// Metadata of main-pass chunk `item` (row item / ipr, piece item % ipr);
// `hint` is the position of a nearby earlier item (or -1).
template <class P>
__device__ __forceinline__ void plan_chunk(const P& prob, const PosTables& tab, int n_pos,
                                           unsigned item, int& hint, PlanRec& rec) {
  StageMeta& mt = rec.s.m;
  ResMeta& rm = rec.s.r;
  const int row = static_cast<int>(item / prob.ipr);
  const int chunk = static_cast<int>(item % prob.ipr);
  const int pos = find_pos(tab.rstart, n_pos, row, hint);
  hint = pos;
  mt.item = static_cast<int>(item);
  mt.pos = pos;
  mt.el_base = chunk * prob.chunk_el;
  mt.n_el = min(prob.chunk_el, prob.V - mt.el_base);
  mt.src2 = nullptr;
  rm.slot = row * prob.ipr + chunk;
  prob.fill_stage(tab, row - tab.rstart[pos], mt, rm);
  rm.item = mt.item;
  mt.slot = rm.slot;
  rm.kind = mt.kind;
  rm.c_hi = mt.c_hi;
  rm.c_lo = mt.c_lo;
}

template <class P>
__device__ void producer_loop(const P& prob, Shared& sh, const PosTables& tab,
                              unsigned char* stages) {
  WsHeader* hdr = prob.ws.hdr;
  int* err = &hdr->error;
  const int lane = threadIdx.x & 31;
  const int n_pos = sh.n_pos;
  const int n_rows = tab.rstart[n_pos];
  const unsigned n_items = static_cast<unsigned>(n_rows) * static_cast<unsigned>(prob.ipr);
  int it = 0;                 // ring position

  // Put a planned chunk into the ring; executed by the one lane holding the
  // record: wait for the slot, store the metadata (16-byte stores, no loads),
  // publish it and start the bulk copies.
  auto issue_own = [&](const PlanRec& rec, int at) {
    const int stage = at % kStages;
    const int rs = at % kResSlots;
    if (at >= kStages) wait_or_flag(sh, &sh.empty[stage], ((at / kStages) - 1) & 1, err);
    if (at >= kResSlots) wait_or_flag(sh, &sh.res_free[rs], ((at / kResSlots) - 1) & 1, err);
    uint4* dm = reinterpret_cast<uint4*>(&sh.meta[stage]);
#pragma unroll
    for (int q = 0; q < kStageWords; ++q) dm[q] = rec.v[q];
    uint4* dr = reinterpret_cast<uint4*>(&sh.res_meta[rs]);
#pragma unroll
    for (int q = 0; q < kResWords16; ++q) dr[q] = rec.v[kStageWords + q];
    mbar_arrive(&sh.res_done[rs]);
    const StageMeta& m = rec.s.m;
    if (prob.bulk) {
      // one or two row pieces of n_el elements: [0, half) and [half, 2 half)
      const uint32_t bytes = static_cast<uint32_t>(m.n_el * prob.es);
      unsigned char* dst = stages + static_cast<size_t>(stage) * kChunkBytes;
      if (!SV_CHECK(bulk_args_ok(dst, m.src, bytes) &&
                        bytes <= static_cast<uint32_t>(m.src2 ? kChunkBytes / 2 : kChunkBytes) &&
                        (m.src2 == nullptr || bulk_args_ok(dst + kChunkBytes / 2, m.src2, bytes)),
                    err)) {
        mbar_arrive(&sh.full[stage]);  // nothing copied: the stage completes empty
        return;
      }
      mbar_arrive_expect_tx(&sh.full[stage], m.src2 ? 2u * bytes : bytes);
      if (m.src2 == nullptr) {
        bulk_copy_g2s_hint(dst, m.src, bytes, &sh.full[stage], policy_evict_first());
      } else {
        bulk_copy_g2s(dst, m.src, bytes, &sh.full[stage]);
        bulk_copy_g2s(dst + kChunkBytes / 2, m.src2, bytes, &sh.full[stage]);
      }
    } else {
      mbar_arrive(&sh.full[stage]);
    }
  };

  // Draw-pass chunks planned by the scout wait in the shared mailbox.  The
  // lane that issues the next ring position first moves every waiting record
  // into the ring, then its own chunk.  The ring position and the mailbox
  // head live in shared memory, so consecutive positions are handed from
  // lane to lane with one __syncwarp and no other warp-wide operation (a
  // collective per chunk measurably slowed the producer).  Only shared
  // memory is read here: the producer never waits on global memory.
  auto issue_mailbox = [&](int at) -> int {  // one lane; returns the next position
    if constexpr (P::kHasDraws) {
      const unsigned t = vload(sh.mb_tail);
      unsigned h = vload(sh.mb_head);
      if (t != h) {
        __threadfence_block();  // the records before their use
        for (; h != t; ++h) {
          PlanRec r;
          const uint4* src = reinterpret_cast<const uint4*>(&sh.mb[h % kMbCap]);
#pragma unroll
          for (int q = 0; q < kStageWords + kResWords16; ++q) r.v[q] = src[q];
          __threadfence_block();
          *reinterpret_cast<volatile unsigned*>(&sh.mb_head) = h + 1u;
          issue_own(r, at++);
        }
      }
    }
    return at;
  };

  // Main pass: this CTA's share (chunks blockIdx.x + j G over the G
  // streaming CTAs), worked out 32 at a time, one chunk per lane and held
  // in that lane's registers, then issued in order, each by its own lane.
  const unsigned G = gridDim.x - n_ctrl_of(prob);
  for (unsigned base = blockIdx.x; base < n_items; base += 32u * G) {
    const int cnt = static_cast<int>(min(32u, (n_items - base + G - 1u) / G));
    PlanRec rec;
    int hint = -1;
    if (lane < cnt) plan_chunk(prob, tab, n_pos, base + static_cast<unsigned>(lane) * G, hint, rec);
    for (int k = 0; k < cnt; ++k) {
      if (lane == k) {
        int at = static_cast<int>(vload(sh.p_it));
        at = issue_mailbox(at);
        issue_own(rec, at);
        *reinterpret_cast<volatile unsigned*>(&sh.p_it) = static_cast<unsigned>(at + 1);
      }
      // ring positions are issued strictly in order: no lane goes on to
      // the next position before this one is in the ring
      __syncwarp();
    }
  }

  if constexpr (P::kHasDraws) {
    // The rest of the draw pass (lane 0): move the scout's records until it
    // is done.
    if (lane == 0) {
      int at = static_cast<int>(vload(sh.p_it));
      uint64_t t0 = 0;
      unsigned backoff = 32;
      for (;;) {
        const int before = at;
        at = issue_mailbox(at);
        if (at != before) {
          t0 = 0;
          backoff = 32;
          continue;
        }
        if (vload(sh.sc_done) != 0u) {
          __threadfence_block();
          if (vload(sh.mb_tail) == vload(sh.mb_head)) break;
          continue;
        }
        const uint64_t now = globaltimer_ns();
        if (t0 == 0) t0 = now;
        if (now - t0 > 2 * wait_limit(sh)) {
          flag_timeout(sh, err);
          break;
        }
        __nanosleep(backoff);
        backoff = min(backoff * 2u, 256u);
      }
      *reinterpret_cast<volatile unsigned*>(&sh.p_it) = static_cast<unsigned>(at);
    }
    __syncwarp();
  }
  it = static_cast<int>(vload(sh.p_it));

  // end of stream: one sentinel per consumer group (the bookkeeper stops at
  // the first)
  if (lane == 0) {
    for (int k = 0; k < kGroups; ++k, ++it) {
      const int stage = it % kStages;
      const int rs = it % kResSlots;
      if (it >= kStages) wait_or_flag(sh, &sh.empty[stage], ((it / kStages) - 1) & 1, err);
      if (it >= kResSlots) wait_or_flag(sh, &sh.res_free[rs], ((it / kResSlots) - 1) & 1, err);
      sh.meta[stage].item = -1;
      sh.res_meta[rs].item = -1;
      mbar_arrive(&sh.res_done[rs]);
      mbar_arrive(&sh.full[stage]);
    }
  }
  __syncwarp();
}

// The draw scout (lane 0 of its warp): walks this CTA's draw-pass claims,
// waits for each claimed draw to be published, plans the chunk and leaves
// the record in the shared mailbox for the producer.  Claim g is chunk
// g % ipr2 of the draw at position g / ipr2 (sampled requests hold the
// first positions, in the order their rows stream).  The claims continue
// the main pass's round robin: claim g goes to the streaming CTA that
// main-pass item n_items + g would go to, so every CTA streams the same
// number of chunks, to within one, and no counter is shared.  The scout
// polls each draw's record itself; a failed request's draw has no chunks
// (the last of its claims clears the record).  All its waits on global
// memory happen here, off the producer's path.
template <class P>
__device__ void scout_loop(const P& prob, Shared& sh, const PosTables& tab) {
  if constexpr (P::kHasDraws) {
    const int lane = threadIdx.x & 31;
    int* err = &prob.ws.hdr->error;
    const unsigned cap = static_cast<unsigned>(sh.n_draw_cap);
    const unsigned G = gridDim.x - n_ctrl_of(prob);
    const unsigned n_claims = cap * static_cast<unsigned>(prob.ipr2);
    const unsigned n_items =
        static_cast<unsigned>(tab.rstart[sh.n_pos]) * static_cast<unsigned>(prob.ipr);
    if (lane == 0 && cap > 0) {
      unsigned tail = 0;
      unsigned cached_d = 0xffffffffu;
      int cached = 0;  // 1: a draw, 0: the request failed
      P2Job job{};
      // the first claim g with (n_items + g) % G == this CTA
      const unsigned first = (blockIdx.x + G - n_items % G) % G;
      for (unsigned g = first; g < n_claims; g += G) {
        // room in the mailbox
        if (tail - vload(sh.mb_head) >= static_cast<unsigned>(kMbCap)) {
          const uint64_t t0 = globaltimer_ns();
          bool ok = true;
          while (tail - vload(sh.mb_head) >= static_cast<unsigned>(kMbCap)) {
            if (globaltimer_ns() - t0 > wait_limit(sh)) {
              ok = false;
              break;
            }
            __nanosleep(64);
          }
          if (!ok) {
            flag_timeout(sh, err);
            break;
          }
        }
        const unsigned d = g / static_cast<unsigned>(prob.ipr2);
        if (d != cached_d) {
          cached = prob.poll_job(tab, static_cast<int>(d), wait_limit(sh), job);
          if (cached < 0) {
            flag_timeout(sh, err);
            break;
          }
          cached_d = d;
        }
        if (cached == 0) {  // a failed request's draw has no chunks
          prob.failed_claim(tab, static_cast<int>(d));
          continue;
        }
        PlanRec rec;
        StageMeta& mt = rec.s.m;
        ResMeta& rm = rec.s.r;
        mt.item = 0x7fffffff;
        mt.pos = -1;
        mt.src2 = nullptr;
        prob.fill_resid(job, static_cast<int>(g % static_cast<unsigned>(prob.ipr2)), mt, rm);
        rm.item = mt.item;
        mt.slot = rm.slot;
        rm.kind = mt.kind;
        rm.c_hi = mt.c_hi;
        rm.c_lo = mt.c_lo;
        uint4* dst = reinterpret_cast<uint4*>(&sh.mb[tail % kMbCap]);
#pragma unroll
        for (int q = 0; q < kStageWords + kResWords16; ++q) dst[q] = rec.v[q];
        __threadfence_block();
        ++tail;
        *reinterpret_cast<volatile unsigned*>(&sh.mb_tail) = tail;
      }
    }
    if (lane == 0) {
      __threadfence_block();
      *reinterpret_cast<volatile unsigned*>(&sh.sc_done) = 1u;
    }
    __syncwarp();
  }
}

template <class P>
__device__ void consumer_loop(const P& prob, Shared& sh, unsigned char* stages) {
  int* err = &prob.ws.hdr->error;
  const int group = (threadIdx.x - kConsBase) / kGroupThreads;
  const int ctid = (threadIdx.x - kConsBase) % kGroupThreads;  // 0 .. kGroupThreads-1
  const int warp = ctid >> 5, lane = ctid & 31;
  for (int j = group;; j += kGroups) {
    const int stage = j % kStages;
    const int rs = j % kResSlots;
    wait_or_flag(sh, &sh.full[stage], (j / kStages) & 1, err);
    const StageMeta mt = sh.meta[stage];
    if (mt.item < 0) {
      if (lane == 0) mbar_arrive(&sh.res_done[rs]);
      break;
    }
    const unsigned char* sp = stages + static_cast<size_t>(stage) * kChunkBytes;
    const float4 part = prob.consume(mt, sp, &sh.empty[stage], ctid, lane);
    if (lane == 0) {
      sh.res_part[rs][warp] = part;
      mbar_arrive(&sh.res_done[rs]);  // release: the partial is visible to the bookkeeper
    }
  }
}

// The bookkeeper: per result slot, combine the consumer warps' partials,
// store them, and append the chunk's ticket to the booked queue.  It never
// waits on global memory, so the result ring keeps moving.
template <class P>
__device__ void bookkeeper_loop(const P& prob, Shared& sh) {
  int* err = &prob.ws.hdr->error;
  const int lane = threadIdx.x & 31;
  for (int j = 0;; ++j) {
    const int rs = j % kResSlots;
    wait_or_flag(sh, &sh.res_done[rs], (j / kResSlots) & 1, err);
    const ResMeta rm = sh.res_meta[rs];
    if (rm.item < 0) break;
    const float4 p = lane < kGroupWarps ? sh.res_part[rs][lane]
                                        : make_float4(kNegInf, 0.f, 0.f, 0.f);
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh.res_free[rs]);
    if constexpr (P::kCtrl) {
      // Control CTAs poll: the results go straight to the workspace, as
      // words the pollers check themselves.  No count, no fence, no queue,
      // nothing waits here.
      if (rm.kind == KIND_RESID_PASS) {
        if constexpr (P::kHasDraws)
          if (lane < kGroupWarps) prob.store_segsums_warp(rm.slot, lane, p);
      } else {
        float2 tot;
        if (rm.kind == KIND_ARGMAX) {
          const VI v = warp_reduce_vi(VI{p.x, lane < kGroupWarps ? __float_as_int(p.y)
                                                                 : 0x7fffffff});
          tot = make_float2(v.v, __int_as_float(v.i));
        } else {
          const MS v = warp_reduce_ms(MS{p.x, p.y}, Scale2{rm.c_hi, rm.c_lo});
          tot = make_float2(v.m, v.s);
        }
        if (lane == 0) prob.store_partial(rm.slot, rm.kind, tot);
      }
      continue;
    }
    {
      float2 tot;
      if (rm.kind == KIND_ARGMAX) {
        const VI v = warp_reduce_vi(VI{p.x, lane < kGroupWarps ? __float_as_int(p.y)
                                                               : 0x7fffffff});
        tot = make_float2(v.v, __int_as_float(v.i));
      } else {
        const MS v = warp_reduce_ms(MS{p.x, p.y}, Scale2{rm.c_hi, rm.c_lo});
        tot = make_float2(v.m, v.s);
      }
      if (lane == 0) prob.ws.partials[rm.slot] = tot;
    }
    __syncwarp();  // every lane's stores before lane 0 publishes the entry
    if (lane == 0) {
      const unsigned t = sh.bq_tail;
      if (t - vload(sh.bq_head) >= static_cast<unsigned>(kBqCap)) {
        const uint64_t t0 = globaltimer_ns();
        while (t - vload(sh.bq_head) >= static_cast<unsigned>(kBqCap)) {
          if (globaltimer_ns() - t0 > wait_limit(sh)) {
            flag_timeout(sh, err);
            break;
          }
          __nanosleep(64);
        }
      }
      sh.bq[t % kBqCap] = make_int4(rm.tkt, rm.need, rm.fin_code, 0);
      __threadfence_block();
      *reinterpret_cast<volatile unsigned*>(&sh.bq_tail) = t + 1u;
    }
  }
  if (lane == 0) {
    __threadfence_block();
    *reinterpret_cast<volatile unsigned*>(&sh.bk_done) = 1u;
  }
  __syncwarp();
}

// Append the codes of the lanes with `done` to the finalize list (ticket
// warp only; all lanes call it): waits, bounded, while the list is full.
__device__ __forceinline__ void fin_push(Shared& sh, bool done, int code, int lane, int* err) {
  const unsigned dmask = __ballot_sync(0xffffffffu, done);
  if (!dmask) return;
  const unsigned ft = vload(sh.fin_tail);
  const unsigned need_room = ft + __popc(dmask);
  if (need_room - vload(sh.fin_claim) > static_cast<unsigned>(kFinCap)) {
    const uint64_t t0 = globaltimer_ns();
    while (need_room - vload(sh.fin_claim) > static_cast<unsigned>(kFinCap)) {
      __nanosleep(200);
      if (globaltimer_ns() - t0 > kWaitLimitNs) {
        if (lane == 0) record_error(err, 0x10);
        break;
      }
    }
  }
  if (done)
    reinterpret_cast<volatile int*>(sh.fin_q)[(ft + __popc(dmask & ((1u << lane) - 1u))) %
                                               kFinCap] = code;
  __syncwarp();
  if (lane == 0) {
    __threadfence_block();
    *reinterpret_cast<volatile unsigned*>(&sh.fin_tail) = need_room;
  }
  __syncwarp();
}

// The ticket warp: first puts this CTA's share of the requests that need no
// main-pass rows (positions blockIdx.x + j G) on the finalize list; then
// takes booked chunks in batches of up to 32 (lane i one chunk), makes
// their partials visible GPU-wide, bumps their tickets and puts each
// request or draw whose ticket completes on the finalize list.  The fence
// and the atomics' round trip happen here, off the result ring.
template <class P>
__device__ void ticketer_loop(const P& prob, Shared& sh, const PosTables& tab) {
  int* err = &prob.ws.hdr->error;
  const int lane = threadIdx.x & 31;
  if constexpr (P::kHasDirectFin && !P::kCtrl) {
    const int G = static_cast<int>(gridDim.x);
    for (int p0 = static_cast<int>(blockIdx.x); p0 < sh.n_pos; p0 += 32 * G) {
      const int p = p0 + lane * G;
      fin_push(sh, p < sh.n_pos && prob.direct_fin(tab, p), p, lane, err);
    }
  }
  unsigned head = 0;
  uint64_t idle_since = 0;
  unsigned backoff = 32;
  for (;;) {
    unsigned tail = vload(sh.bq_tail);
    if (tail == head) {
      if (vload(sh.bk_done) != 0u) {
        __threadfence_block();
        tail = vload(sh.bq_tail);
        if (tail == head) break;
      } else {
        const uint64_t now = globaltimer_ns();
        if (idle_since == 0) idle_since = now;
        if (now - idle_since > 2 * kWaitLimitNs) {
          if (lane == 0) record_error(err, 0x10);
          break;
        }
        __nanosleep(backoff);
        backoff = min(backoff * 2u, 256u);
        continue;
      }
    }
    idle_since = 0;
    backoff = 32;
    __threadfence_block();  // the entries (and the bookkeeper's stores) before reading them
    const int nb = static_cast<int>(min(tail - head, 32u));
    const int4 e = lane < nb ? sh.bq[(head + lane) % kBqCap] : make_int4(0, 0, 0, 0);
    {
      fence_acq_rel_gpu();  // the partials (stored by the bookkeeper) -> GPU scope before the tickets
      bool done = false;
      if (lane < nb) {
        const unsigned old = atomic_add_acq_rel(&prob.ws.tickets[e.x], 1u);
        done = old + 1u == static_cast<unsigned>(e.y);
      }
      fin_push(sh, done, e.z, lane, err);
    }
    head += static_cast<unsigned>(nb);
    __syncwarp();
    if (lane == 0) *reinterpret_cast<volatile unsigned*>(&sh.bq_head) = head;
  }
  if (lane == 0) {
    __threadfence_block();
    *reinterpret_cast<volatile unsigned*>(&sh.tk_done) = 1u;
  }
  __syncwarp();
}

// Take the next finalize-list entry: returns it, -2 when the CTA is done,
// -1 when there is nothing yet.  Marks the caller busy while it holds one.
__device__ __forceinline__ int fin_take(Shared& sh) {
  const unsigned c = vload(sh.fin_claim);
  if (c != vload(sh.fin_tail)) {
    atomicAdd(&sh.fin_busy, 1u);
    if (atomicCAS(&sh.fin_claim, c, c + 1u) == c) {
      __threadfence_block();
      return reinterpret_cast<volatile int*>(sh.fin_q)[c % kFinCap];
    }
    atomicSub(&sh.fin_busy, 1u);
    return -1;
  }
  if (vload(sh.tk_done) != 0u && vload(sh.fin_claim) == vload(sh.fin_tail)) return -2;
  return -1;
}

__device__ __forceinline__ void fin_release(Shared& sh) {
  __threadfence_block();
  atomicSub(&sh.fin_busy, 1u);
}

template <class P>
__device__ void finalizer_loop(const P& prob, Shared& sh, const PosTables& tab) {
  const int ftid = threadIdx.x - kFinBase;
  const int fwarp = ftid >> 5, lane = ftid & 31;
  uint64_t idle_since = 0;
  unsigned backoff = 32;
  if constexpr (P::kWarpFinalize) {
    for (;;) {
      int cmd = -1;
      if (lane == 0) {
        cmd = fin_take(sh);
        if (cmd == -1) {
          const uint64_t now = globaltimer_ns();
          if (idle_since == 0) idle_since = now;
          if (now - idle_since > 2 * kWaitLimitNs) {
            record_error(&prob.ws.hdr->error, 0x10);
            cmd = -2;
          }
        } else {
          idle_since = 0;
        }
      }
      cmd = __shfl_sync(0xffffffffu, cmd, 0);
      if (cmd == -2) break;
      if (cmd >= 0) {
        prob.finalize_warp(sh, tab, cmd, lane, sh.wfin[fwarp]);
        __syncwarp();
        if (lane == 0) fin_release(sh);
        backoff = 32;
      } else {
        __nanosleep(backoff);
        backoff = min(backoff * 2u, 256u);
      }
    }
  } else {
    for (;;) {
      if (ftid == 0) {
        int cmd = fin_take(sh);
        if (cmd == -1) {
          const uint64_t now = globaltimer_ns();
          if (idle_since == 0) idle_since = now;
          if (now - idle_since > 2 * kWaitLimitNs) {
            record_error(&prob.ws.hdr->error, 0x10);
            cmd = -2;
          }
          __nanosleep(backoff);
          backoff = min(backoff * 2u, 256u);
        } else {
          idle_since = 0;
          backoff = 32;
        }
        sh.fin_cmd = cmd;
      }
      named_sync(1, kFinThreads);
      const int cmd = sh.fin_cmd;
      named_sync(1, kFinThreads);
      if (cmd == -2) break;
      if (cmd >= 0) {
        prob.finalize(sh, tab, cmd, ftid);
        if (ftid == 0) fin_release(sh);
      }
    }
  }
}

// A control CTA: every warp takes the positions c + n_ctrl (warp + nw k)
// (c = this control CTA's index), waits for each one's rows and finalizes
// it, then waits for the draw passes of the ones that published a draw and
// runs their draw finalizes.  Control CTAs share no SM with the streaming
// roles, so a finalize runs as soon as its last chunk is booked.  The
// per-warp scratch lives in the unused chunk ring.
template <class P>
__device__ void control_loop(const P& prob, Shared& sh, const PosTables& tab,
                             unsigned char* scratch) {
  if constexpr (P::kCtrl) {
    constexpr int nw = kThreads / 32;
    const int warp = static_cast<int>(threadIdx.x) >> 5, lane = threadIdx.x & 31;
    const int n_ctrl = prob.n_ctrl;
    const int c = static_cast<int>(blockIdx.x) - (static_cast<int>(gridDim.x) - n_ctrl);
    WarpFin& wf = reinterpret_cast<WarpFin*>(scratch)[warp];
    const int first = c + n_ctrl * warp, step = n_ctrl * nw;
    unsigned long long drew = 0ull;  // positions of this warp that published a draw
    int k = 0;
    for (int p = first; p < sh.n_pos; p += step, ++k)
      if (prob.ctrl_request(sh, tab, p, lane, wf) && k < 64) drew |= 1ull << k;
    k = 0;
    for (int p = first; p < sh.n_pos && k < 64; p += step, ++k)
      if ((drew >> k) & 1ull) prob.ctrl_draw(sh, tab, p, lane, wf);
  }
}

template <class P>
__global__ void __launch_bounds__(kThreads, 1) verify_kernel(const P prob) {
  static_assert(kThreads / 32 * sizeof(WarpFin) <= static_cast<size_t>(kStages) * kChunkBytes,
                "control CTAs keep one warp scratch per warp in the chunk ring");
  static_assert(!P::kHasDraws || P::kWarpFinalize,
                "the draw scout takes a finalizer warp: group finalizes need all four");
  extern __shared__ __align__(1024) unsigned char smem_dyn[];
  // Launched with programmatic stream serialisation: wait for the previous
  // work on the stream (which may have produced the inputs, and used the
  // same workspace) before touching global memory, and let the next launch
  // start filling SMs as this one drains.
  if (threadIdx.x < 32) prob.prefetch_args(threadIdx.x);
  grid_dependency_wait();
  grid_launch_dependents();
  // 128-byte aligned base (the launch adds 128 bytes of slack)
  unsigned char* smem_raw = smem_dyn + ((128u - (smem_u32(smem_dyn) & 127u)) & 127u);
  unsigned char* stages = smem_raw;
  Shared& sh = *reinterpret_cast<Shared*>(smem_raw + kStages * kChunkBytes);
  unsigned char* tail = smem_raw + kStages * kChunkBytes + ((shared_bytes<P>() + 15) & ~size_t(15));
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
      mbar_init(&sh.empty[s], kGroupWarps);
    }
    for (int s = 0; s < kResSlots; ++s) {
      mbar_init(&sh.res_done[s], kGroupWarps + 1);
      mbar_init(&sh.res_free[s], 1);
    }
    fence_mbar_init();
    sh.timed_out = 0;
    sh.fin_claim = sh.fin_tail = sh.fin_busy = 0u;
    sh.bk_done = 0u;
    sh.bq_tail = sh.bq_head = 0u;
    sh.tk_done = 0u;
    sh.p_it = 0u;
    if constexpr (P::kHasDraws) sh.mb_tail = sh.mb_head = sh.sc_done = 0u;
    sh.fin_cmd = -1;
    sh.n_draw_cap = 0;
  }
  prob.preamble(sh, tab, scan_tmp, stages);
  __syncthreads();

  if (P::kCtrl && blockIdx.x >= gridDim.x - n_ctrl_of(prob)) {
    control_loop(prob, sh, tab, stages);
  } else if (threadIdx.x < kBkBase) {
    producer_loop(prob, sh, tab, stages);
  } else if (threadIdx.x < kTkBase) {
    bookkeeper_loop(prob, sh);
  } else if (threadIdx.x < kFinBase) {
    if (!P::kCtrl) ticketer_loop(prob, sh, tab);  // control CTAs poll the data words themselves
  } else if (threadIdx.x < kConsBase) {
    if (P::kHasDraws && threadIdx.x >= kScBase) scout_loop(prob, sh, tab);
    else if (!P::kCtrl) finalizer_loop(prob, sh, tab);
  } else {
    consumer_loop(prob, sh, stages);
  }
  // Nothing to reset at the end: every word of the workspace this call
  // wrote is cleared by the role that read it last (partials by their
  // finalize, segment sums and draw records by the draw finalize, a failed
  // draw's record by its last claim), so a CTA just exits.
}

}  // namespace sv
