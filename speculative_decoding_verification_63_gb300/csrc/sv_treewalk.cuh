// sv_treewalk.cuh -- token-tree verification as a walk on a thread-block
// cluster, one request per cluster.
//
// The tree of each request is depth-first linearised with parent indices
// (CMU 15-779 Lecture 17 notes, "Speculative Decoding", sec. 4.3).  The walk
// starts at the root: VerifyGreedy for t == 0 (sec. 4.4), multi-step
// speculative sampling for t > 0 (sec. 4.5): the children of the current
// node are tried in ascending index order against the residual r (initially
// p_node); child c is accepted iff u_c q_c(x_c) < r(x_c), otherwise
// r <- norm(max(0, r - q_c)); all rejected: a draw from r with u_sample; a
// node without children: a draw from p_node (the bonus token).  Two more
// stochastic rules share the walk: children drawn without replacement (the
// j-th child is tested against q_j = q with the earlier siblings' tokens
// removed and renormalised, sec. 4.5 and sec. 10 exercise 7), and naive
// sampling (draw x from p_node with the node's own uniform; move to the
// first child whose token is x, else emit x).
//
// The walk only ever needs the rows on its path: the target row of each
// node it stands on and the draft rows its children are tested against.
// So it reads those rows, lazily, and nothing else.  The CL CTAs of the
// cluster hold contiguous slices of the vocabulary (rank r: tokens
// [r Ls, (r+1) Ls)); each CTA keeps the slices of the rows in use, and of
// the rows the next step may need (prefetched with 1-D bulk copies), in a
// small row cache in shared memory, and the residual r of its slice in fp32
// (two buffers: a rejection that leaves no mass keeps the old r).  Every
// decision is taken after an exchange: each CTA reduces its slice, writes a
// 32-byte record, the cluster synchronises, and every CTA reads the CL
// records from the others' shared memory and merges them in rank order --
// so all CTAs hold the same values and take the same branches.
//   node start  (max, sum 2^((x - m) c)) of p_node and of the first child's
//               draft row, and the logits of the child's token (its owner);
//   accept      u_c q(x_c) < r(x_c) in fp64 from the merged values;
//   rejection   r <- max(0, r - q_c) over the slice, the slice's mass and,
//               for the next child, its draft row's statistics and the
//               logits / residual at its token, in one exchange;
//   draw        weights in token order (fp32 within a thread, float pairs
//               across threads and CTAs), one exchange of the slice totals,
//               the CTA whose slice holds u S finds the token, one more
//               exchange hands it to every CTA.
#pragma once

#include "sv_cluster.cuh"
#include "sv_rowpass.cuh"

namespace sv {

constexpr int kTwThreads = 512;
constexpr int kTwWarps = kTwThreads / 32;
constexpr int kTwSlots = 6;         // row slices cached per CTA
constexpr int kTwMaxNodes = 64;     // = SV_MAX_TREE_NODES
constexpr int kTwMaxCl = 16;

struct TreeWalkProblem {
  int B, N, M, V, max_depth, es, mode;
  int Ls;          // slice length (tokens), a multiple of 16 / es
  int slot_bytes;  // bytes of one cached row slice (a multiple of 128)
  bool bulk;       // rows and strides fit for 1-D bulk copies
  const char* target;
  int64_t t_stride;  // bytes
  const char* draft;
  int64_t d_stride;
  const int* tokens;
  const int* parent;
  const int* q_row;
  const int* num_nodes;
  const float* temperature;
  const int* top_k;
  const float* u_accept;
  const float* u_sample;
  int* out_tokens;
  int* out_len;
  int* accept_len;
  int* accepted_nodes;
  WsHeader* hdr;
};

struct TwShared {
  uint64_t bar[kTwSlots];     // one per cached row slice
  int tag[kTwSlots];          // (b << 17 | kind << 16 | row) + 1, 0: empty
  unsigned issued[kTwSlots];  // loads issued into the slot
  int par[kTwMaxNodes], tok[kTwMaxNodes], qr[kTwMaxNodes], depth[kTwMaxNodes];
  int ch_start[kTwMaxNodes + 1], ch_list[kTwMaxNodes];
  int path[kTwMaxNodes];
  uint4 xr[2][2];             // this CTA's exchange record (double-buffered)
  uint4 xall[kTwMaxCl][2];    // the cluster's records of the last exchange
  float red[4][kTwWarps];     // block-reduction scratch
  int redf[kTwWarps];
  float ua[kTwMaxNodes];      // the request's accept uniforms, and its sample uniform
  float us;
  DF dscan[kTwWarps];
  int ibuf[4];
  int err;
  int timed_out;
};

__device__ __forceinline__ uint64_t tw_limit(const TwShared& sh) {
  return sh.timed_out ? kWaitLimitAfterTimeoutNs : kWaitLimitNs;
}

template <int ES>
__device__ __forceinline__ float tw_elem(const unsigned char* slot, int e) {
  if constexpr (ES == 2) return bf16_bits_to_float(reinterpret_cast<const uint16_t*>(slot)[e]);
  else return reinterpret_cast<const float*>(slot)[e];
}

// Block (kTwThreads) reduction of (max, sum) pairs; every thread gets it.
__device__ __forceinline__ MS tw_block_ms(MS v, Scale2 c, TwShared& sh) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  v = warp_reduce_ms(v, c);
  __syncthreads();
  if (lane == 0) {
    sh.red[0][warp] = v.m;
    sh.red[1][warp] = v.s;
  }
  __syncthreads();
  MS w = lane < kTwWarps ? MS{sh.red[0][lane], sh.red[1][lane]} : MS{kNegInf, 0.f};
  w = warp_reduce_ms(w, c);
  return w;
}

// Two block (max, sum) reductions and an OR of flags with one exchange
// through shared memory; each pair combines exactly as tw_block_ms would.
__device__ __forceinline__ int tw_block_ms2(MS& a, MS& b, int flag, Scale2 c, TwShared& sh) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  a = warp_reduce_ms(a, c);
  b = warp_reduce_ms(b, c);
  flag = __reduce_or_sync(0xffffffffu, flag);
  __syncthreads();
  if (lane == 0) {
    sh.red[0][warp] = a.m;
    sh.red[1][warp] = a.s;
    sh.red[2][warp] = b.m;
    sh.red[3][warp] = b.s;
    sh.redf[warp] = flag;
  }
  __syncthreads();
  const bool in = lane < kTwWarps;
  a = warp_reduce_ms(in ? MS{sh.red[0][lane], sh.red[1][lane]} : MS{kNegInf, 0.f}, c);
  b = warp_reduce_ms(in ? MS{sh.red[2][lane], sh.red[3][lane]} : MS{kNegInf, 0.f}, c);
  return __reduce_or_sync(0xffffffffu, in ? sh.redf[lane] : 0);
}

__device__ __forceinline__ VI tw_block_vi(VI v, TwShared& sh) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  v = warp_reduce_vi(v);
  __syncthreads();
  if (lane == 0) {
    sh.red[0][warp] = v.v;
    sh.red[1][warp] = __int_as_float(v.i);
  }
  __syncthreads();
  VI w = lane < kTwWarps ? VI{sh.red[0][lane], __float_as_int(sh.red[1][lane])}
                         : VI{kNegInf, 0x7fffffff};
  return warp_reduce_vi(w);
}

__device__ __forceinline__ float tw_block_sum(float x, TwShared& sh, int row) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  __syncthreads();
  if (lane == 0) sh.red[row][warp] = x;
  __syncthreads();
  float w = lane < kTwWarps ? sh.red[row][lane] : 0.f;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) w += __shfl_xor_sync(0xffffffffu, w, o);
  return w;
}

__device__ __forceinline__ int tw_block_max_int(int x, TwShared& sh) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = max(x, __shfl_xor_sync(0xffffffffu, x, o));
  __syncthreads();
  if (lane == 0) sh.red[3][warp] = __int_as_float(x);
  __syncthreads();
  int w = lane < kTwWarps ? __float_as_int(sh.red[3][lane]) : -1;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) w = max(w, __shfl_xor_sync(0xffffffffu, w, o));
  return w;
}

// Block inclusive / exclusive scan of float pairs in thread order.
__device__ __forceinline__ DF tw_block_scan_df(DF x, TwShared& sh, DF& excl, DF& total) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const DF inc = warp_incl_scan_df(x, lane);
  DF ex{__shfl_up_sync(0xffffffffu, inc.hi, 1), __shfl_up_sync(0xffffffffu, inc.lo, 1)};
  if (lane == 0) ex = DF{0.f, 0.f};
  __syncthreads();
  if (lane == 31) sh.dscan[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    const DF w = lane < kTwWarps ? sh.dscan[lane] : DF{0.f, 0.f};
    const DF wi = warp_incl_scan_df(w, lane);
    __syncwarp();
    if (lane < kTwWarps) sh.dscan[lane] = wi;
  }
  __syncthreads();
  const DF off = warp > 0 ? sh.dscan[warp - 1] : DF{0.f, 0.f};
  total = sh.dscan[kTwWarps - 1];
  excl = df_add(off, ex);
  return df_add(off, inc);
}

template <int ES>
__global__ void __launch_bounds__(kTwThreads, 1) tree_walk_kernel(const TreeWalkProblem P) {
  extern __shared__ __align__(128) unsigned char tw_smem[];
  __shared__ __align__(16) TwShared sh;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cl_rank(), CL = cl_size(), cid = cl_id(), nC = cl_count();
  const int N = P.N, V = P.V;
  const int lo = static_cast<int>(rank) * P.Ls;
  const int n_sl = max(0, min(P.Ls, V - lo));
  // dynamic shared memory: kTwSlots row slices, then two fp32 residual slices
  unsigned char* slots = tw_smem;
  float* wres0 = reinterpret_cast<float*>(tw_smem + static_cast<size_t>(kTwSlots) * P.slot_bytes);
  float* wres1 = wres0 + ((P.Ls + 31) & ~31);

  if (tid == 0) {
    for (int s = 0; s < kTwSlots; ++s) {
      mbar_init(&sh.bar[s], 1);
      sh.tag[s] = 0;
      sh.issued[s] = 0u;
    }
    fence_mbar_init();
    sh.timed_out = 0;
  }
  grid_dependency_wait();
  grid_launch_dependents();
  __syncthreads();
  const uint64_t pol = policy_evict_first();
  int xpar = 0;  // exchange parity (every CTA takes the same exchanges)

  // ---- the exchange: thread 0's record to the cluster; afterwards every
  // thread can read all CL records in sh.xall (rank order)
  auto exchange = [&](uint4 a, uint4 b) {
    if (tid == 0) {
      sh.xr[xpar][0] = a;
      sh.xr[xpar][1] = b;
    }
    cl_sync();
    if (warp == 0 && lane < static_cast<int>(CL)) {
      const uint32_t ad = cl_map(&sh.xr[xpar][0], static_cast<uint32_t>(lane));
      sh.xall[lane][0] = cl_ld_u4(ad);
      sh.xall[lane][1] = cl_ld_u4(ad + 16);
    }
    xpar ^= 1;
    __syncthreads();
  };
  auto flag_timeout = [&]() {
    sh.timed_out = 1;
    record_error(&P.hdr->error, SV_DERR_TIMEOUT);
  };

  // ---- row cache: kind 0 target row (b, n), kind 1 draft row (b, m); a
  // cluster walks several requests in turn, so the key holds b as well
  int cur_b = 0;
  auto key_of = [&](int kind, int row) { return ((cur_b << 17) | (kind << 16) | row) + 1; };
  auto find_slot = [&](int key) {
    int f = -1;
#pragma unroll
    for (int s2 = kTwSlots - 1; s2 >= 0; --s2)
      if (sh.tag[s2] == key) f = s2;
    return f;
  };
  // warp 0, every lane: make sure the row slice is in (or on its way into) a
  // slot, evicting a slot whose key is not in protect[0..np); lane s looks
  // at slot s
  auto ensure = [&](int b, int kind, int row, const int* protect, int np) {
    const int key = key_of(kind, row);
    const int tg = lane < kTwSlots ? sh.tag[lane] : -1;
    if (__ballot_sync(0xffffffffu, tg == key)) return;
    bool keep = lane >= kTwSlots;
    for (int q = 0; q < np; ++q) keep |= tg == protect[q];
    const unsigned cand = __ballot_sync(0xffffffffu, !keep);
    if (!cand) return;  // nothing evictable: it will be loaded on demand
    const int s = __ffs(cand) - 1;
    const char* src = kind == 0
        ? P.target + (static_cast<int64_t>(b) * N + row) * P.t_stride + static_cast<int64_t>(lo) * ES
        : P.draft + (static_cast<int64_t>(b) * P.M + row) * P.d_stride + static_cast<int64_t>(lo) * ES;
    unsigned char* dst = slots + static_cast<size_t>(s) * P.slot_bytes;
    if (lane == 0) {
      if (sh.issued[s] > 0u &&
          !mbar_wait_bounded(&sh.bar[s], (sh.issued[s] - 1u) & 1u, tw_limit(sh)))
        flag_timeout();  // the previous load has to land before the slot is reused
      sh.tag[s] = key;
      sh.issued[s] += 1u;
    }
    __syncwarp();
    if (P.bulk) {
      if (lane == 0) {
        const uint32_t bytes = static_cast<uint32_t>(n_sl * ES);
        if (bytes > 0 && !SV_CHECK(bulk_args_ok(dst, src, bytes) && bytes <= static_cast<uint32_t>(P.slot_bytes),
                                   &P.hdr->error)) {
          mbar_arrive(&sh.bar[s]);  // nothing copied: the slot completes empty
        } else {
          mbar_arrive_expect_tx(&sh.bar[s], bytes);
          if (bytes > 0) bulk_copy_g2s_hint(dst, src, bytes, &sh.bar[s], pol);
        }
      }
    } else {
      // rows unfit for bulk copies: the warp copies the slice
      for (int e = lane; e < n_sl; e += 32) {
        if constexpr (ES == 2)
          reinterpret_cast<uint16_t*>(dst)[e] = reinterpret_cast<const uint16_t*>(src)[e];
        else
          reinterpret_cast<uint32_t*>(dst)[e] = reinterpret_cast<const uint32_t*>(src)[e];
      }
      __threadfence_block();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.bar[s]);
    }
    __syncwarp();
  };
  // all threads: the slot of a row, once loaded.  The caller has passed a
  // barrier since the cache table last changed, so every thread finds the
  // same slot; a row that found no slot when it was prefetched is asked for
  // now (anything but the rows of the current step, ibuf[0..1], may make
  // room), between two barriers.
  auto acquire = [&](int b, int kind, int row) -> const unsigned char* {
    int s = find_slot(key_of(kind, row));
    if (s < 0) {
      __syncthreads();  // every thread has read the table
      if (warp == 0) {
        const int keep[2] = {sh.ibuf[0], sh.ibuf[1]};
        ensure(b, kind, row, keep, 2);
      }
      __syncthreads();
      s = find_slot(key_of(kind, row));
      if (s < 0) return nullptr;
    }
    if (!mbar_wait_bounded(&sh.bar[s], (sh.issued[s] - 1u) & 1u, tw_limit(sh)) && tid == 0)
      flag_timeout();
    return slots + static_cast<size_t>(s) * P.slot_bytes;
  };

  // warp 0: the rows wanted next (lane i < nw holds the i-th by priority:
  // kind, row) put on their way into the cache, all at once, one lane per
  // row.  A slot is reused only when its key is not wanted and its last load
  // has landed, so nothing here waits; a wanted row left without a slot is
  // loaded by acquire when it is needed.
  auto prefetch = [&](int b, int nw, int wkind, int wrow) {
    const int wkey = lane < nw ? key_of(wkind, wrow) : -2;
    const int tg = lane < kTwSlots ? sh.tag[lane] : -3;
    const bool idle = lane < kTwSlots &&
                      (sh.issued[lane] == 0u ||
                       mbar_test_wait(&sh.bar[lane], (sh.issued[lane] - 1u) & 1u));
    bool present = false, wanted = false;
#pragma unroll
    for (int q = 0; q < kTwSlots; ++q) {
      // both shuffles run in every lane (never inside a short-circuit)
      const int tq = __shfl_sync(0xffffffffu, tg, q);
      const int wq = __shfl_sync(0xffffffffu, wkey, q);
      present |= lane < nw && tq == wkey;              // in a slot already
      present |= lane < nw && q < lane && wq == wkey;  // an earlier lane asks for it
      wanted |= q < nw && tg == wq;                    // slot `lane` holds a wanted row
    }
    const unsigned free_m = __ballot_sync(0xffffffffu, lane < kTwSlots && !wanted && idle);
    const unsigned miss_m = __ballot_sync(0xffffffffu, lane < nw && !present);
    int slot = -1;
    if ((miss_m >> lane) & 1u) {
      unsigned f = free_m;
      for (int q = __popc(miss_m & ((1u << lane) - 1u)); q > 0 && f; --q) f &= f - 1u;
      if (f) slot = __ffs(f) - 1;
    }
    const char* src = nullptr;
    if (slot >= 0)
      src = wkind == 0 ? P.target + (static_cast<int64_t>(b) * N + wrow) * P.t_stride +
                             static_cast<int64_t>(lo) * ES
                       : P.draft + (static_cast<int64_t>(b) * P.M + wrow) * P.d_stride +
                             static_cast<int64_t>(lo) * ES;
    if (slot >= 0) {
      sh.tag[slot] = wkey;
      sh.issued[slot] += 1u;
      if (P.bulk) {
        const uint32_t bytes = static_cast<uint32_t>(n_sl * ES);
        unsigned char* dst = slots + static_cast<size_t>(slot) * P.slot_bytes;
        if (bytes > 0 && !SV_CHECK(bulk_args_ok(dst, src, bytes) && bytes <= static_cast<uint32_t>(P.slot_bytes),
                                   &P.hdr->error)) {
          mbar_arrive(&sh.bar[slot]);  // nothing copied: the slot completes empty
        } else {
          mbar_arrive_expect_tx(&sh.bar[slot], bytes);
          if (bytes > 0) bulk_copy_g2s_hint(dst, src, bytes, &sh.bar[slot], pol);
        }
      }
    }
    __syncwarp();
    if (!P.bulk) {
      // rows unfit for bulk copies: the warp copies the slices in turn
      unsigned m = __ballot_sync(0xffffffffu, slot >= 0);
      while (m) {
        const int i = __ffs(m) - 1;
        m &= m - 1u;
        const int si = __shfl_sync(0xffffffffu, slot, i);
        const char* sp = reinterpret_cast<const char*>(
            __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(src), i));
        unsigned char* dst = slots + static_cast<size_t>(si) * P.slot_bytes;
        for (int e = lane; e < n_sl; e += 32) {
          if constexpr (ES == 2)
            reinterpret_cast<uint16_t*>(dst)[e] = reinterpret_cast<const uint16_t*>(sp)[e];
          else
            reinterpret_cast<uint32_t*>(dst)[e] = reinterpret_cast<const uint32_t*>(sp)[e];
        }
        __threadfence_block();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.bar[si]);
      }
    }
    __syncwarp();
  };

  for (int b = static_cast<int>(cid); b < P.B; b += static_cast<int>(nC)) {
    cur_b = b;
    // the root's target row is needed whatever the tree holds: on its way now
    if (warp == 0) {
      const int prot[1] = {key_of(0, 0)};
      ensure(b, 0, 0, prot, 1);
    }
    // ---- the request's tree, checked identically in every CTA
    const int nn = P.num_nodes ? P.num_nodes[b] : N;
    const float t = P.temperature[b];
    const int tk = P.top_k ? P.top_k[b] : 0;
    const bool greedy = t == 0.f;
    const bool naive = P.mode == kTreeNaive && !greedy;
    const bool use_q = !greedy && !naive;
    if (tid < N) {
      sh.par[tid] = P.parent[static_cast<size_t>(b) * N + tid];
      sh.tok[tid] = P.tokens[static_cast<size_t>(b) * N + tid];
      sh.qr[tid] = P.q_row[static_cast<size_t>(b) * N + tid];
      sh.ua[tid] = greedy ? 0.f : P.u_accept[static_cast<size_t>(b) * N + tid];
    }
    if (tid == 0) sh.us = greedy ? 0.f : P.u_sample[b];
    if (tid == 0) {
      int e0 = 0;
      if (nn < 1 || nn > N || !(t >= 0.f) || tk < 0) e0 |= SV_DERR_ARG;
      else if (!greedy && tk > 0 && tk < V) e0 |= SV_DERR_ARG;  // top-k trees: not supported
      else if (use_q && nn > 1 && P.draft == nullptr) e0 |= SV_DERR_ARG;
      sh.err = e0;
    }
    __syncthreads();
    if (sh.err == 0 && tid < nn) {
      // node n: its parent, token and draft row, its depth (walking up), and
      // how many children it has
      const int n = tid;
      int e1 = 0;
      if (n == 0) {
        if (sh.par[0] != -1) e1 |= SV_DERR_TREE;
      } else {
        const int p = sh.par[n];
        if (p < 0 || p >= n || (use_q && (sh.qr[n] < 0 || sh.qr[n] >= P.M))) e1 |= SV_DERR_TREE;
        else if (sh.tok[n] < 0 || sh.tok[n] >= V) e1 |= SV_DERR_TOKEN;
      }
      int d = 0, x = n;
      while (x > 0 && d <= P.max_depth) {
        const int px = sh.par[x];
        if (px < 0 || px >= x) break;
        x = px;
        ++d;
      }
      if (d > P.max_depth) e1 |= SV_DERR_TREE;
      sh.depth[n] = d;
      int cnt = 0;
      for (int c2 = n + 1; c2 < nn; ++c2) cnt += sh.par[c2] == n;
      sh.ch_start[n + 1] = cnt;
      if (e1) atomicOr(&sh.err, e1);
    }
    __syncthreads();
    if (sh.err == 0) {
      // children lists in ascending index (CSR): counts scanned, then every
      // node writes itself after its earlier siblings
      if (warp == 0) {
        // ch_start[n + 1] holds node n's count: an inclusive scan (two per lane)
        const int n0 = 2 * lane + 1, n1 = 2 * lane + 2;
        const int a0 = n0 <= nn ? sh.ch_start[n0] : 0, a1 = n1 <= nn ? sh.ch_start[n1] : 0;
        const unsigned inc = warp_incl_scan_u(static_cast<unsigned>(a0 + a1), lane);
        const int ex = static_cast<int>(inc) - (a0 + a1);
        __syncwarp();
        if (n0 <= nn) sh.ch_start[n0] = ex + a0;
        if (n1 <= nn) sh.ch_start[n1] = ex + a0 + a1;
        if (lane == 0) sh.ch_start[0] = 0;
      }
      __syncthreads();
      if (tid >= 1 && tid < nn) {
        const int p = sh.par[tid];
        int before = 0;
        for (int c2 = p + 1; c2 < tid; ++c2) before += sh.par[c2] == p;
        sh.ch_list[sh.ch_start[p] + before] = tid;
      }
    }
    __syncthreads();
    int err = sh.err;
    const Scale2 c = scale_for(t);
    const double cd = static_cast<double>(c.hi) + static_cast<double>(c.lo);
    int node = 0, L = 0, token = -1;

    // weights of the draw over this CTA's slice: mode 0 = 2^((l - mp) c) of
    // the row slice `row`, mode 1 = the residual buffer `wr`
    auto weight = [&](int mode, const unsigned char* row, const float* wr, float mp, int e) {
      if (e >= n_sl) return 0.f;
      if (mode == 1) return wr[e];
      return fast_exp2(scaled_arg(tw_elem<ES>(row, e), mp, c));
    };
    // the inverse-CDF draw with uniform u; the token in every CTA (-1: no mass)
    auto draw = [&](int mode, const unsigned char* row, const float* wr, float mp, float u) -> int {
      const int G = (n_sl + kTwThreads - 1) / kTwThreads;
      const int e0 = tid * G;
      float ts = 0.f;
      int last = -1;
      for (int e = e0; e < min(e0 + G, n_sl); ++e) {
        const float w = weight(mode, row, wr, mp, e);
        ts = __fadd_rn(ts, w);
        if (w > 0.f) last = lo + e;
      }
      DF ex, tot;
      const DF inc = tw_block_scan_df(DF{ts, 0.f}, sh, ex, tot);
      const int lmax = tw_block_max_int(last, sh);
      exchange(make_uint4(__float_as_uint(tot.hi), __float_as_uint(tot.lo), static_cast<unsigned>(lmax), 0u),
               make_uint4(0u, 0u, 0u, 0u));
      // merged in rank order, identically everywhere
      DF S{0.f, 0.f};
      for (int r = 0; r < static_cast<int>(CL); ++r)
        S = df_add(S, DF{__uint_as_float(sh.xall[r][0].x), __uint_as_float(sh.xall[r][0].y)});
      const DF target = df_mul(u, S);
      int owner = -1, fb = -1;
      DF Pw{0.f, 0.f}, run{0.f, 0.f};
      for (int r = 0; r < static_cast<int>(CL); ++r) {
        const DF Sr{__uint_as_float(sh.xall[r][0].x), __uint_as_float(sh.xall[r][0].y)};
        const DF nx = df_add(run, Sr);
        if (owner < 0 && Sr.hi > 0.f && df_lt(target, nx)) {
          owner = r;
          Pw = run;
        }
        if (static_cast<int>(sh.xall[r][0].z) >= 0) fb = static_cast<int>(sh.xall[r][0].z);
        run = nx;
      }
      int tok = -1;
      if (S.hi > 0.f) {
        if (owner < 0) {
          tok = fb;  // rounding left u S at the end: the last positive weight
        } else if (static_cast<int>(rank) == owner) {
          if (tid == 0) sh.ibuf[2] = 0x7fffffff;
          __syncthreads();
          if (ts > 0.f && df_lt(target, df_add(Pw, inc))) atomicMin(&sh.ibuf[2], tid);
          __syncthreads();
          if (tid == sh.ibuf[2]) {
            DF cc = df_add(Pw, ex);
            int found = -1, lastp = -1;
            for (int e = e0; e < min(e0 + G, n_sl) && found < 0; ++e) {
              const float w = weight(mode, row, wr, mp, e);
              cc = df_add(cc, w);
              if (w > 0.f) lastp = lo + e;
              if (w > 0.f && df_lt(target, cc)) found = lo + e;
            }
            sh.ibuf[3] = found >= 0 ? found : lastp;
          }
          __syncthreads();
          tok = sh.ibuf[2] == 0x7fffffff ? static_cast<int>(sh.xall[rank][0].z) : sh.ibuf[3];
        }
        // the owner hands the token to the cluster
        exchange(make_uint4(static_cast<unsigned>(tok), 0u, 0u, 0u), make_uint4(0u, 0u, 0u, 0u));
        if (owner >= 0) tok = static_cast<int>(sh.xall[owner][0].x);
      }
      return tok;
    };

    while (!err) {
      const int c0 = sh.ch_start[node], nc = sh.ch_start[node + 1] - c0;
      // rows now and, prefetched, for the next step: the children's target
      // rows (and for MSS their children's draft rows)
      if (warp == 0) {
        int nw = 0, wkind = -1, wrow = -1;
        auto want = [&](int kd, int rw) {
          if (nw < kTwSlots) {
            if (lane == nw) {
              wkind = kd;
              wrow = rw;
            }
            ++nw;
          }
        };
        want(0, node);
        if (use_q && nc > 0) want(1, sh.qr[sh.ch_list[c0]]);
        if (lane == 0) {
          sh.ibuf[0] = key_of(0, node);
          sh.ibuf[1] = use_q && nc > 0 ? key_of(1, sh.qr[sh.ch_list[c0]]) : sh.ibuf[0];
        }
        for (int k = 0; k < nc && nw < kTwSlots; ++k) {
          const int ch = sh.ch_list[c0 + k];
          want(0, ch);
          if (use_q) {
            const int g0 = sh.ch_start[ch], gn = sh.ch_start[ch + 1] - g0;
            if (gn > 0) want(1, sh.qr[sh.ch_list[g0]]);
          }
        }
        prefetch(b, nw, wkind, wrow);
      }
      __syncthreads();  // the cache table, for acquire
      const unsigned char* prow = acquire(b, 0, node);
      if (greedy) {
        // ---- VerifyGreedy: the argmax of p_node (lowest id on ties)
        VI v{kNegInf, 0x7fffffff};
        bool bad = false;
        for (int e = tid; e < n_sl; e += kTwThreads) {
          const float x = tw_elem<ES>(prow, e);
          if (x != x || x == kPosInf) bad = true;
          if (x > v.v) v = VI{x, lo + e};
        }
        v = tw_block_vi(v, sh);
        const int fl = __syncthreads_or(bad) ? SV_DERR_NONFINITE : 0;
        exchange(make_uint4(__float_as_uint(v.v), static_cast<unsigned>(v.i), static_cast<unsigned>(fl), 0u),
                 make_uint4(0u, 0u, 0u, 0u));
        VI m{kNegInf, 0x7fffffff};
        int f2 = 0;
        for (int r = 0; r < static_cast<int>(CL); ++r) {
          m = vi_better(m, VI{__uint_as_float(sh.xall[r][0].x), static_cast<int>(sh.xall[r][0].y)});
          f2 |= static_cast<int>(sh.xall[r][0].z);
        }
        if (!f2 && m.v == kNegInf) f2 |= SV_DERR_MASS;
        if (f2) {
          err |= f2;
          break;
        }
        int next = -1;
        for (int k = 0; k < nc; ++k)
          if (sh.tok[sh.ch_list[c0 + k]] == m.i) {
            next = sh.ch_list[c0 + k];
            break;
          }
        if (next < 0) {
          token = m.i;
          break;
        }
        if (tid == 0) sh.path[L] = next;
        ++L;
        node = next;
        continue;
      }

      // ---- p_node's statistics (and, for MSS, the first child's draft row
      // and the logits of its token)
      const unsigned char* qrow = nullptr;
      int qrow_id = -1;
      if (use_q && nc > 0) {
        qrow_id = sh.qr[sh.ch_list[c0]];
        qrow = acquire(b, 1, qrow_id);
      }
      float mloc[2] = {kNegInf, kNegInf};
      bool bad = false;
      for (int e = tid; e < n_sl; e += kTwThreads) {
        const float x = tw_elem<ES>(prow, e);
        bad |= x != x || x == kPosInf;
        mloc[0] = fmaxf(mloc[0], x);
        if (qrow) {
          const float y = tw_elem<ES>(qrow, e);
          bad |= y != y || y == kPosInf;
          mloc[1] = fmaxf(mloc[1], y);
        }
      }
      float sloc[2] = {0.f, 0.f};
      for (int e = tid; e < n_sl; e += kTwThreads) {
        if (mloc[0] != kNegInf) sloc[0] += fast_exp2(scaled_arg(tw_elem<ES>(prow, e), mloc[0], c));
        if (qrow && mloc[1] != kNegInf) sloc[1] += fast_exp2(scaled_arg(tw_elem<ES>(qrow, e), mloc[1], c));
      }
      MS bp{mloc[0], sloc[0]}, bq{mloc[1], sloc[1]};
      const int fl0 = tw_block_ms2(bp, bq, bad ? 1 : 0, c, sh) ? SV_DERR_NONFINITE : 0;
      if (!qrow) bq = MS{kNegInf, 0.f};
      float gp = kNegInf, gq = kNegInf;
      int own = 0;
      if (nc > 0 && !naive) {
        const int x = sh.tok[sh.ch_list[c0]];
        if (x >= lo && x < lo + n_sl) {
          own = 0x100;
          gp = tw_elem<ES>(prow, x - lo);
          if (qrow) gq = tw_elem<ES>(qrow, x - lo);
        }
      }
      exchange(make_uint4(__float_as_uint(bp.m), __float_as_uint(bp.s), __float_as_uint(bq.m),
                          __float_as_uint(bq.s)),
               make_uint4(__float_as_uint(gp), __float_as_uint(gq), static_cast<unsigned>(fl0 | own), 0u));
      MS mp{kNegInf, 0.f}, mq{kNegInf, 0.f};
      int f2 = 0;
      for (int r = 0; r < static_cast<int>(CL); ++r) {
        const int fr = static_cast<int>(sh.xall[r][1].z);
        f2 |= fr;
        if (fr & 0x100) {
          gp = __uint_as_float(sh.xall[r][1].x);
          gq = __uint_as_float(sh.xall[r][1].y);
        }
        mp = ms_combine(mp, MS{__uint_as_float(sh.xall[r][0].x), __uint_as_float(sh.xall[r][0].y)}, c);
        mq = ms_combine(mq, MS{__uint_as_float(sh.xall[r][0].z), __uint_as_float(sh.xall[r][0].w)}, c);
      }
      f2 &= ~0x100;
      if (!f2 && (mp.m == kNegInf || !(mp.s > 0.f))) f2 |= SV_DERR_MASS;
      if (!f2 && qrow && (mq.m == kNegInf || !(mq.s > 0.f))) f2 |= SV_DERR_MASS;
      if (f2) {
        err |= f2;
        break;
      }

      if (naive) {
        // ---- naive sampling: x ~ p_node with the node's own uniform
        const int x = draw(0, prow, nullptr, mp.m, sh.ua[node]);
        if (x < 0) {
          err |= SV_DERR_MASS;
          break;
        }
        int next = -1;
        for (int k = 0; k < nc; ++k)
          if (sh.tok[sh.ch_list[c0 + k]] == x) {
            next = sh.ch_list[c0 + k];
            break;
          }
        if (next < 0) {
          token = x;
          break;
        }
        if (tid == 0) sh.path[L] = next;
        ++L;
        node = next;
        continue;
      }
      if (nc == 0) {
        // ---- a leaf: the bonus token from p_node
        token = draw(0, prow, nullptr, mp.m, sh.us);
        if (token < 0) err |= SV_DERR_MASS;
        break;
      }

      // ---- multi-step speculative sampling over the children
      // r = p_node (rstate 0) or wres[cur] / S (rstate 1)
      int rstate = 0, cur = 0;
      double invS = 0.0;   // 1 / S in fp64 (thread 0: the accept tests)
      float finvS = 0.f;    // 1 / S in fp32 (every thread: the residual passes)
      float Sres = 0.f;     // S, the residual's mass, in every thread
      int next = -1;
      int nq_id = qrow_id;        // the draft row whose statistics are in mq
      for (int k = 0; k < nc; ++k) {
        const int ch = sh.ch_list[c0 + k];
        const int x = sh.tok[ch];
        const int row_id = sh.qr[ch];
        // The accept test.  Every thread holds the same merged values, so
        // every thread takes the same fp32 decision; the calls it leaves open
        // (close ones, exponents below -96) and the rule without
        // replacement after the first child (q_j = q off the earlier
        // siblings' distinct tokens, scaled by 1 / (1 - R), R their q mass)
        // go to thread 0, which decides them as below and hands the result
        // to the block.
        int acc = -1;
        float fqs = 1.f;
        if (!(P.mode == kTreeNoReplace && k > 0)) {
          const float u32 = sh.ua[ch];
          float ahp = 0.f, ahq = 0.f;
          const float nq32 = exp2_scaled_pair(gq, mq.m, c, ahq);
          const float num32 = rstate == 0 ? exp2_scaled_pair(gp, mp.m, c, ahp) : gp;
          const float den32 = rstate == 0 ? mp.s : Sres;
          const float lhs = u32 * nq32 * den32, rhs = num32 * mq.s;
          if (ahp >= -96.f && ahq >= -96.f && fabsf(lhs - rhs) > 4e-6f * fmaxf(lhs, rhs))
            acc = lhs < rhs;
        }
        if (acc < 0) {
        if (tid == 0) {
          double qs = 1.0;
          bool removed = false;
          if (P.mode == kTreeNoReplace && k > 0) {
            const char* qg = P.draft + (static_cast<int64_t>(b) * P.M + row_id) * P.d_stride;
            double R = 0.0;
            for (int j = 0; j < k; ++j) {
              const int y = sh.tok[sh.ch_list[c0 + j]];
              bool dup = false;
              for (int i2 = 0; i2 < j; ++i2) dup |= sh.tok[sh.ch_list[c0 + i2]] == y;
              if (dup) continue;
              removed |= y == x;
              R += exp2_nonpos((static_cast<double>(load_logit(qg, ES, y)) - mq.m) * cd) /
                   static_cast<double>(mq.s);
            }
            qs = R < 1.0 ? 1.0 / (1.0 - R) : 0.0;
          }
          // u q(x) < r(x) with q = nq qs / Zq and r = np / Zp (r = p_node) or
          // r = w / S (a residual), taken without divisions: u nq qs D < N Zq
          // with (N, D) = (np, Zp) or (w, S).  First in fp32 with the
          // exponents as float pairs (about 5e-7 relative); calls closer than
          // 4e-6 relative, and exponents below -96, in fp64.
          const float u32 = sh.ua[ch];
          float ahp = 0.f, ahq = 0.f;
          const float nq32 = removed ? 0.f : exp2_scaled_pair(gq, mq.m, c, ahq);
          const float num32 = rstate == 0 ? exp2_scaled_pair(gp, mp.m, c, ahp) : gp;
          const float den32 = rstate == 0 ? mp.s : sh.red[2][1];
          const float lhs = u32 * (nq32 * static_cast<float>(qs)) * den32, rhs = num32 * mq.s;
          int a0;
          if (ahp >= -96.f && ahq >= -96.f && qs == 1.0 &&
              fabsf(lhs - rhs) > 4e-6f * fmaxf(lhs, rhs)) {
            a0 = lhs < rhs;
          } else {
            const double q = removed ? 0.0
                                     : exp2_nonpos((static_cast<double>(gq) - mq.m) * cd) /
                                           static_cast<double>(mq.s) * qs;
            const double r = rstate == 0
                                 ? exp2_nonpos((static_cast<double>(gp) - mp.m) * cd) /
                                       static_cast<double>(mp.s)
                                 : static_cast<double>(gp) * invS;
            a0 = static_cast<double>(u32) * q < r;
          }
          sh.ibuf[2] = a0;
          sh.red[2][0] = static_cast<float>(qs);
        }
        __syncthreads();
        acc = sh.ibuf[2];
        fqs = sh.red[2][0];
        __syncthreads();
        }
        const bool accept = acc != 0;
        if (accept) {
          next = ch;
          break;
        }
        // rejected: r <- max(0, r - q_j) into the other buffer; for the next
        // child its draft row's statistics and the values at its token
        const unsigned char* qcur = acquire(b, 1, row_id);
        const int nxt = cur ^ 1;
        float* wout = nxt ? wres1 : wres0;
        const float* win = cur ? wres1 : wres0;
        const float izp = rcp_fma(mp.s), izq = rcp_fma(mq.s);
        float part = 0.f;
        for (int e = tid; e < n_sl; e += kTwThreads) {
          const float rt = rstate == 0 ? fast_exp2(scaled_arg(tw_elem<ES>(prow, e), mp.m, c)) * izp
                                       : win[e] * finvS;
          const float qt = fast_exp2(scaled_arg(tw_elem<ES>(qcur, e), mq.m, c)) * izq * fqs;
          const float w = fmaxf(rt - qt, 0.f);
          wout[e] = w;
          part += w;
        }
        __syncthreads();
        float fix = 0.f;
        if (P.mode == kTreeNoReplace && k > 0 && tid == 0) {
          // q_j is 0 on the removed tokens: the residual there is r itself
          for (int j = 0; j < k; ++j) {
            const int y = sh.tok[sh.ch_list[c0 + j]];
            bool dup = false;
            for (int i2 = 0; i2 < j; ++i2) dup |= sh.tok[sh.ch_list[c0 + i2]] == y;
            if (dup || y < lo || y >= lo + n_sl) continue;
            const int e = y - lo;
            const float ry = rstate == 0 ? fast_exp2(scaled_arg(tw_elem<ES>(prow, e), mp.m, c)) * izp
                                         : win[e] * finvS;
            fix += ry - wout[e];  // the slice's mass changes by the put-back value
            wout[e] = ry;
          }
        }
        const float S_loc = tw_block_sum(part + fix, sh, 0);
        // the next child: its draft row (statistics if it differs) and the
        // owner's values at its token
        const bool more = k + 1 < nc;
        const int ch2 = more ? sh.ch_list[c0 + k + 1] : -1;
        const int x2 = more ? sh.tok[ch2] : -1;
        const int row2 = more ? sh.qr[ch2] : -1;
        const bool new_row = more && row2 != nq_id;
        const unsigned char* q2 = new_row ? acquire(b, 1, row2) : qcur;
        MS b2{kNegInf, 0.f};
        bool bad2 = false;
        if (new_row) {
          float m2 = kNegInf;
          for (int e = tid; e < n_sl; e += kTwThreads) {
            const float y = tw_elem<ES>(q2, e);
            bad2 |= y != y || y == kPosInf;
            m2 = fmaxf(m2, y);
          }
          float s2 = 0.f;
          if (m2 != kNegInf)
            for (int e = tid; e < n_sl; e += kTwThreads) s2 += fast_exp2(scaled_arg(tw_elem<ES>(q2, e), m2, c));
          bad2 = __syncthreads_or(bad2);
          b2 = tw_block_ms(MS{m2, s2}, c, sh);
        }
        float gw = kNegInf, gq2 = kNegInf;
        int own2 = 0;
        if (more && x2 >= lo && x2 < lo + n_sl) {
          own2 = 0x100;
          gw = wout[x2 - lo];                        // the new residual
          gq2 = tw_elem<ES>(q2, x2 - lo);
        }
        // the old r at x2 as well (kept when the new residual has no mass)
        float gold = kNegInf;
        if (more && own2) {
          const int e = x2 - lo;
          gold = rstate == 0 ? tw_elem<ES>(prow, e) : win[e];
        }
        exchange(make_uint4(__float_as_uint(S_loc), __float_as_uint(b2.m), __float_as_uint(b2.s),
                            __float_as_uint(gold)),
                 make_uint4(__float_as_uint(gw), __float_as_uint(gq2),
                            static_cast<unsigned>((bad2 ? SV_DERR_NONFINITE : 0) | own2), 0u));
        float S = 0.f;  // the mass in fp32 (its sign decides; 1/S goes through fp64 once)
        MS m2{kNegInf, 0.f};
        int f3 = 0;
        float gw_m = kNegInf, gq_m = kNegInf, gold_m = kNegInf;
        for (int r = 0; r < static_cast<int>(CL); ++r) {
          S += __uint_as_float(sh.xall[r][0].x);
          m2 = ms_combine(m2, MS{__uint_as_float(sh.xall[r][0].y), __uint_as_float(sh.xall[r][0].z)}, c);
          const int fr = static_cast<int>(sh.xall[r][1].z);
          f3 |= fr;
          if (fr & 0x100) {
            gw_m = __uint_as_float(sh.xall[r][1].x);
            gq_m = __uint_as_float(sh.xall[r][1].y);
            gold_m = __uint_as_float(sh.xall[r][0].w);
          }
        }
        f3 &= ~0x100;
        if (new_row && !f3 && (m2.m == kNegInf || !(m2.s > 0.f))) f3 |= SV_DERR_MASS;
        if (f3) {
          err |= f3;
          break;
        }
        if (S > 0.f) {
          // r <- w / S (a residual of zero mass, by rounding only, keeps r)
          rstate = 1;
          cur = nxt;
          finvS = rcp_fma(S);
          Sres = S;
          if (tid == 0) {
            invS = 1.0 / static_cast<double>(S);
            sh.red[2][1] = S;  // read by thread 0 only (the next accept test)
          }
          gp = gw_m;
        } else {
          gp = gold_m;  // r unchanged: its value at the next token
        }
        if (new_row) {
          mq = m2;
          nq_id = row2;
        }
        gq = gq_m;
      }
      if (err) break;
      if (next >= 0) {
        if (tid == 0) sh.path[L] = next;
        ++L;
        node = next;
        continue;
      }
      // ---- every child rejected: the draw from r with u_sample
      token = rstate == 0 ? draw(0, prow, nullptr, mp.m, sh.us)
                          : draw(1, nullptr, cur ? wres1 : wres0, 0.f, sh.us);
      if (token < 0) err |= SV_DERR_MASS;
      break;
    }

    // ---- outputs (rank 0)
    __syncthreads();
    if (rank == 0) {
      const int D = P.max_depth;
      for (int i = tid; i <= D; i += kTwThreads) {
        int v = -1;
        if (!err) {
          if (i < L) v = sh.tok[sh.path[i]];
          else if (i == L) v = token;
        }
        P.out_tokens[static_cast<size_t>(b) * (D + 1) + i] = v;
      }
      for (int i = tid; i < D; i += kTwThreads)
        P.accepted_nodes[static_cast<size_t>(b) * D + i] = (!err && i < L) ? sh.path[i] : -1;
      if (tid == 0) {
        P.out_len[b] = err ? 0 : L + 1;
        P.accept_len[b] = err ? 0 : L;
        if (err) record_error(&P.hdr->error, err);
      }
    }
    __syncthreads();
  }
  // the cached slices' loads have landed before the CTA leaves
  if (tid == 0)
    for (int s = 0; s < kTwSlots; ++s)
      if (sh.issued[s] > 0u) mbar_wait_bounded(&sh.bar[s], (sh.issued[s] - 1u) & 1u, tw_limit(sh));
  __syncthreads();
  cl_sync();
}

}  // namespace sv
