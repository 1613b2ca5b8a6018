// ep_route.cu -- routing-map kernels of ep_prepare (sm_103a).
//
// What prepare computes (TransformerEngine PR #3034, "Expert Parallelism:
// common C API + NCCL EP backend", section "Per-step (allocation-free,
// CUDA-graph capturable)", nvte_ep_prepare): per-expert token counts and a
// routing map, each expert block padded to dispatch_output_per_expert_alignment.
// On one GPU there is no routing all-gather; the map is built in place.
//
//   c_e   = number of routes (t,k) with topk_idx[t,k] == e
//   p_e   = roundup(c_e, A),  off_e = p_0 + ... + p_{e-1},  P = off_E
//   slot  = off_e + (number of earlier routes, in (t,k) order, to expert e)
//
// Route r = t*K + k.  The routes are cut into contiguous chunks (one per CTA)
// and each chunk into contiguous per-warp ranges, so "earlier" is: earlier
// chunk, then earlier warp, then earlier 32-route step, then lower lane.  The
// lane part comes from a peer mask of the lanes holding the same expert (one
// ballot per bit of the expert id) and a population count of the lower lanes;
// the warp part from per-warp counters in
// shared memory; the chunk part from an exclusive scan over chunks.  No atomics
// decide an order, so every slot is the unique stable one.
//
// Two shapes:
//   cluster: one launch of a thread-block cluster of up to 16 CTAs (8 where
//            the device cannot run a 16-CTA cluster).  Each CTA counts its
//            chunk, the CTAs read each other's per-expert totals through
//            distributed shared memory, each computes the aligned offsets, and
//            each assigns the slots of its chunk (decode to DeepSeek-V3-sized
//            batches);
//   chunked: ep_route_hist (per-chunk counts) -> ep_route_scan (one warp per
//            expert scans over chunks; the last CTA to finish does the aligned
//            scan over experts and the padding list) -> ep_route_assign
//            (slots), for batches beyond the cluster's reach and for the
//            fixed-scratch entry point.
#include <cooperative_groups.h>

#include <algorithm>
#include <mutex>

#include "ep_internal.cuh"

namespace ep {
namespace {

namespace cg = cooperative_groups;
constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ int decode_expert(long long v, int E, int& bad) {
  if (v >= 0 && v < E) return static_cast<int>(v);
  if (v != -1) bad = 1;  // outside [-1, E): treated as masked, flagged
  return -1;
}

// Largest expert count whose warp steps use __match_any_sync for the peer
// mask (see warp_assign).
constexpr int kMatchAnyMaxExperts = 16;

// Bits that tell the keys 0..E apart (E stands for "no expert").
__device__ __forceinline__ int key_bits(int E) { return 32 - __clz(E); }

// Lanes of the warp whose key equals this lane's: one ballot per key bit, each
// lane keeping the lanes that agree with it on every bit.  Same result as
// __match_any_sync, at a cost that does not grow with the number of distinct
// keys in the warp (used above kMatchAnyMaxExperts experts).
__device__ __forceinline__ unsigned peer_mask(int key, int nbits) {
  unsigned m = kFull;
  for (int b = 0; b < nbits; ++b) {
    const int bit = (key >> b) & 1;
    const unsigned bal = __ballot_sync(kFull, bit);
    m &= bit ? bal : ~bal;
  }
  return m;
}

// A warp's routes [lo, hi) (at most 32*kMaxJ): route lo + j*32 + lane is held
// by this lane as an int16 expert id (-1 for none) in half j&1 of pk[j/2].
using Packed = unsigned[kMaxJ / 2];

__device__ __forceinline__ int unpack_expert(const Packed& pk, int j) {
  return static_cast<int>(static_cast<short>((pk[j >> 1] >> (16 * (j & 1))) & 0xffffu));
}

// Loads and decodes the warp's routes, 8 independent loads per lane at a
// time so that their latencies overlap, and adds each valid route to the
// warp's counter row (order-free, so a shared-memory atomic suffices).  The
// row belongs to this warp alone: it is zeroed here, while the first loads
// are in flight, and a __syncwarp orders the zeroing before the atomics.
__device__ __forceinline__ void warp_load_count(const long long* __restrict__ idx, int lo, int hi,
                                                int E, int* wrow, Packed& pk, int& bad) {
  const int lane = threadIdx.x & 31;
  const int nj = (hi - lo + 31) >> 5;
#pragma unroll
  for (int jb = 0; jb < kMaxJ; jb += 8) {
    if (jb > 0 && jb >= nj) break;
    long long v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int r = lo + (jb + j) * 32 + lane;
      v[j] = (jb + j < nj && r < hi) ? __ldg(idx + r) : -1LL;
    }
    if (jb == 0) {
      for (int e = lane; e < E; e += 32) wrow[e] = 0;
      __syncwarp();
    }
#pragma unroll
    for (int j = 0; j < 8; j += 2) {
      const int e0 = decode_expert(v[j], E, bad);
      const int e1 = decode_expert(v[j + 1], E, bad);
      if (e0 >= 0) atomicAdd(&wrow[e0], 1);
      if (e1 >= 0) atomicAdd(&wrow[e1], 1);
      pk[(jb + j) >> 1] = (static_cast<unsigned>(e0) & 0xffffu) | (static_cast<unsigned>(e1) << 16);
    }
  }
}

// Slots of the warp's routes, in route order; wbase[e] is the next free row
// of expert e for this warp and advances as routes are placed.  A lane's rank
// among the lanes holding the same expert is the number of such lanes below it.
// With `dest` (sharded layers), the owner rank e / eloc of each route's
// expert is written next to its slot (-1 for a masked route).
// Unrolled: a rolled loop that consumed the packed ids from the front
// measured slower (DeepSeek-V3-sized batch, 16 steps per warp: 12.1K ->
// 13.5K cycles; decode 1.7K -> 1.9K), this part being bound by instruction
// issue rather than by instruction fetch.
__device__ __forceinline__ void warp_assign(const Packed& pk, int lo, int hi, int E, int* wbase,
                                            int* __restrict__ slot, int* __restrict__ dest = nullptr,
                                            int eloc = 1) {
  const int lane = threadIdx.x & 31;
  const unsigned lower = (1u << lane) - 1u;
  const int nbits = key_bits(E);
  const int nj = (hi - lo + 31) >> 5;
#pragma unroll
  for (int j = 0; j < kMaxJ; ++j) {
    if (j >= nj) break;
    const int r = lo + j * 32 + lane;
    const int e = unpack_expert(pk, j);  // -1 beyond hi
    // Few experts: __match_any_sync, whose cost grows with the number of
    // distinct keys in the warp; many: one ballot per key bit.  Measured per
    // 32-route step (clock64 stamps): E=8 (Mixtral-sized batch) 0.45K vs
    // 0.63K cycles; E=256 with 32 distinct experts per step (DeepSeek-V3-
    // sized) 1.05K vs 0.75K.
    const unsigned m = E <= kMatchAnyMaxExperts ? __match_any_sync(kFull, e >= 0 ? e : E)
                                                : peer_mask(e >= 0 ? e : E, nbits);
    int s = -1;
    if (e >= 0) s = wbase[e] + __popc(m & lower);
    __syncwarp();
    if (e >= 0 && lane == __ffs(m) - 1) wbase[e] += __popc(m);
    __syncwarp();
    if (r < hi) {
      slot[r] = s;
      if (dest != nullptr) dest[r] = e >= 0 ? e / eloc : -1;
    }
  }
}

// Column pass over the [W][E] per-warp counter table (W <= kMaxW): for each
// expert (thread-strided), wcnt[w][e] <- base(e) + sum of wcnt[w'][e] over
// w' < w.  The W loads of a column are issued together before any store.
// Returns nothing; with tot != nullptr, tot[e] = the column's sum.
constexpr int kMaxW = 16;

__device__ __forceinline__ void column_prefix(int* wcnt, int W, int E, const int* base0,
                                              const int* base1, int* tot) {
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int v[kMaxW];
#pragma unroll
    for (int w = 0; w < kMaxW; ++w) v[w] = w < W ? wcnt[w * E + e] : 0;
    const int b = (base0 ? base0[e] : 0) + (base1 ? base1[e] : 0);
    int run = b;
#pragma unroll
    for (int w = 0; w < kMaxW; ++w)
      if (w < W) {
        wcnt[w * E + e] = run;
        run += v[w];
      }
    if (tot != nullptr) tot[e] = run - b;
  }
}

// wcnt[w][e] += base0[e] + base1[e] for every warp w.
__device__ __forceinline__ void column_add(int* wcnt, int W, int E, const int* base0,
                                           const int* base1) {
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int b = base0[e] + (base1 ? base1[e] : 0);
    int v[kMaxW];
#pragma unroll
    for (int w = 0; w < kMaxW; ++w) v[w] = w < W ? wcnt[w * E + e] : 0;
#pragma unroll
    for (int w = 0; w < kMaxW; ++w)
      if (w < W) wcnt[w * E + e] = v[w] + b;
  }
}

// Cluster barrier halves (thread-block clusters, sm_90+): arrive with release
// semantics, wait with acquire semantics.  Every thread of every CTA of the
// cluster executes each of them.
__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// c rounded up to a multiple of A (A = 2^a_log2 when a_log2 >= 0: shifts).
__device__ __forceinline__ unsigned roundup(unsigned c, unsigned A, int a_log2) {
  if (a_log2 >= 0) return ((c + A - 1u) >> a_log2) << a_log2;
  return (c + A - 1u) / A * A;
}

// Exclusive scan over the block of (x, y) pairs given per thread in (xs, ys):
// returns the sums over lower threads; *tx, *ty = the block's totals.  Two
// barriers; the caller's next access to `wt` must follow another barrier.
__device__ __forceinline__ void block_scan2(int xs, int ys, int* wt, int* ex, int* ey, int* tx,
                                            int* ty) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int ix = xs, iy = ys;
#pragma unroll 1
  for (int d = 1; d < 32; d <<= 1) {
    const int a = __shfl_up_sync(kFull, ix, d);
    const int b = __shfl_up_sync(kFull, iy, d);
    if (lane >= d) {
      ix += a;
      iy += b;
    }
  }
  if (lane == 31) {
    wt[warp] = ix;
    wt[32 + warp] = iy;
  }
  __syncthreads();
  if (warp == 0) {
    int a = lane < nw ? wt[lane] : 0, b = lane < nw ? wt[32 + lane] : 0;
    const int a0 = a, b0 = b;
#pragma unroll 1
    for (int d = 1; d < 32; d <<= 1) {
      const int u = __shfl_up_sync(kFull, a, d);
      const int v = __shfl_up_sync(kFull, b, d);
      if (lane >= d) {
        a += u;
        b += v;
      }
    }
    wt[64 + lane] = a - a0;
    wt[96 + lane] = b - b0;
    if (lane == 31) {
      wt[128] = a;
      wt[129] = b;
    }
  }
  __syncthreads();
  *ex = wt[64 + warp] + ix - xs;
  *ey = wt[96 + warp] + iy - ys;
  *tx = wt[128];
  *ty = wt[129];
}

// finalize_compute for many experts: every thread takes a run of
// ceil(E / blockDim) experts and a block-wide scan of the run sums gives the
// runs' bases (at 256 experts: 2.6K cycles for one warp over runs of 8).
__device__ void finalize_compute_block(const RouteParams& p, const int* cnt_s, int* off_s,
                                       int* pad_s, int* P_out, int* npad_out) {
  __shared__ int wt[130];
  const int E = p.E;
  const unsigned A = static_cast<unsigned>(p.A);
  const int per = (E + static_cast<int>(blockDim.x) - 1) / static_cast<int>(blockDim.x);
  const int lo = min(static_cast<int>(threadIdx.x) * per, E), hi = min(lo + per, E);
  int sp = 0, sd = 0;
#pragma unroll 1
  for (int e = lo; e < hi; ++e) {
    const unsigned c = static_cast<unsigned>(cnt_s[e]);
    const unsigned pe = roundup(c, A, p.a_log2);
    sp += static_cast<int>(pe);
    sd += static_cast<int>(pe - c);
  }
  int rp, rd, P, npad;
  block_scan2(sp, sd, wt, &rp, &rd, &P, &npad);
#pragma unroll 1
  for (int e = lo; e < hi; ++e) {
    const unsigned c = static_cast<unsigned>(cnt_s[e]);
    const unsigned pe = roundup(c, A, p.a_log2);
    off_s[e] = rp;
    pad_s[e] = rd;
    rp += static_cast<int>(pe);
    rd += static_cast<int>(pe - c);
  }
  if (threadIdx.x == 0) {
    off_s[E] = P;
    pad_s[E] = npad;
  }
  __syncthreads();
  *P_out = P;
  *npad_out = npad;
}

// Given c_e in cnt_s: off_s <- off_e (and off_s[E] = P), pad_s <- the
// exclusive scan of the padding rows per expert (pad_s[E] = their number).
// The loops are kept rolled: this code runs once per launch, and code run
// for the first time in a launch is paid in instruction fetches.  Measured
// with clock64 stamps on GB300: the unrolled 5-step shuffle scan took 2.7K-
// 3.3K cycles the first time and 0.2K when run again in the same launch.
// One warp scans: lane l owns a contiguous run of ceil(E/32) experts, sums it,
// takes the exclusive prefix of the lane sums by shuffles, and writes its
// run's offsets.  The whole CTA calls this (one barrier).
__device__ void finalize_compute(const RouteParams& p, const int* cnt_s, int* off_s, int* pad_s,
                                 int* P_out, int* npad_out) {
  const int E = p.E;
  const unsigned A = static_cast<unsigned>(p.A);
  if (E > 64) {
    finalize_compute_block(p, cnt_s, off_s, pad_s, P_out, npad_out);
    return;
  }
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const int per = (E + 31) / 32;
    const int lo = min(lane * per, E), hi = min(lo + per, E);
    int sp = 0, sd = 0;
#pragma unroll 1
    for (int e = lo; e < hi; ++e) {
      const unsigned c = static_cast<unsigned>(cnt_s[e]);
      const unsigned pe = roundup(c, A, p.a_log2);
      sp += static_cast<int>(pe);
      sd += static_cast<int>(pe - c);
    }
    int ip = sp, id = sd;
#pragma unroll 1
    for (int d = 1; d < 32; d <<= 1) {
      const int y = __shfl_up_sync(kFull, ip, d);
      const int z = __shfl_up_sync(kFull, id, d);
      if (lane >= d) {
        ip += y;
        id += z;
      }
    }
    int rp = ip - sp, rd = id - sd;
#pragma unroll 1
    for (int e = lo; e < hi; ++e) {
      const unsigned c = static_cast<unsigned>(cnt_s[e]);
      const unsigned pe = roundup(c, A, p.a_log2);
      off_s[e] = rp;
      pad_s[e] = rd;
      rp += static_cast<int>(pe);
      rd += static_cast<int>(pe - c);
    }
    if (lane == 31) {
      off_s[E] = ip;
      pad_s[E] = id;
    }
  }
  __syncthreads();
  *P_out = off_s[E];
  *npad_out = pad_s[E];
}

// Writes counts, offsets and the header (part 0), and this part's share of
// the padding list (entries part*blockDim + tid, stride nparts*blockDim).
__device__ void finalize_write(const RouteParams& p, const int* cnt_s, const int* off_s,
                               const int* pad_s, int P, int npad, int bad, int part, int nparts) {
  const int E = p.E;
  if (part == 0) {
    for (int e = threadIdx.x; e <= E; e += blockDim.x) p.offsets[e] = off_s[e];
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
      p.counts[e] = cnt_s[e];
      p.counts_user[e] = cnt_s[e];
    }
    if (threadIdx.x == 0) {
      unsigned st = bad ? EP_ST_BAD_INDEX : 0u;
      if (static_cast<long long>(P) > p.R) st |= EP_ST_OVERFLOW;
      p.hdr[kHdrStatus] = static_cast<int>(st);
      p.hdr[kHdrT] = p.T;
      p.hdr[kHdrP] = P;
      p.hdr[kHdrNPad] = npad;
      p.hdr[kHdrA] = p.A;
      p.hdr[kHdrV] = P - npad;
      p.hdr[kHdrMagic] = kPreparedMagic;
    }
  }
  // Padding rows, ascending: expert e's padding rows off_e + c_e .. off_e +
  // p_e - 1 go to entries pad_s[e] .. pad_s[e+1] - 1, one warp per expert.
  // Skipped when P exceeds the capacity (the row calls then write nothing);
  // otherwise npad <= min(P, E*(A-1)) fits the list.
  if (npad == 0 || static_cast<long long>(P) > p.R || npad > p.pad_cap) return;
  const int lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
  for (int e = part * nwarps + (threadIdx.x >> 5); e < E; e += nparts * nwarps) {
    const int first = off_s[e] + cnt_s[e], n = pad_s[e + 1] - pad_s[e];
    for (int i = lane; i < n; i += 32) p.pad_list[pad_s[e] + i] = first + i;
  }
}

// Shared memory of the cluster kernel, ints: per-warp counters [W][E], this
// CTA's totals [E], lower CTAs' totals [E], counts [E], offsets and padding
// scans [E+1] each, a flag word (+3 pad); the sharded mode adds the counts
// over all ranks [E].
__host__ __device__ constexpr size_t cluster_smem_bytes(int W, int E, bool sharded = false) {
  return static_cast<size_t>(W * E + 3 * E + 2 * (E + 1) + 4 + (sharded ? E : 0)) * 4;
}

// Modes of the cluster kernel: the routing map of a single buffer; this
// rank's histogram only (sharded layers, before the counts are exchanged);
// the routing map of a sharded layer from the all-gathered counts.
enum PrepareMode { kModeLocal = 0, kModeCount = 1, kModeShard = 2 };

// Sharded layers: from the all-gathered counts p.all_counts [N][E] (row r =
// rank r's histogram) and this rank's own counts `mine` [E], computes
//   tall[e]  = routes to e over all ranks;
//   off_s[e] = first row of e's block on its owner (blocks of the owner's
//              experts in expert order from row 0, each padded to A), then,
//              after the outputs are written, the first row of THIS rank's
//              routes in that block: + the routes to e of ranks before it;
//   pad_s[e] = first entry of e's padding rows in its owner's padding list;
// writes, as the owner of experts [rank*E/N, (rank+1)*E/N), the counts, the
// offsets [E/N + 1], the header and the padding list (CTA `part` of `nparts`
// writes its share of the list; part 0 the rest).  Status: BAD_INDEX (this
// rank's indices), OVERFLOW when any owner's rows exceed R, COUNTS_MISMATCH
// when row `rank` of the table is not this rank's histogram.  One warp per
// owner scans its experts: lane l a run of ceil(E/N / 32) of them, then a
// shuffle scan of the run sums.  The whole CTA calls this (three barriers).
__device__ void shard_finalize(const RouteParams& p, const int* mine, int* tall, int* off_s,
                               int* pad_s, int bad, int part, int nparts) {
  const int E = p.E, N = p.nranks, rank = p.rank, eloc = E / N;
  const unsigned A = static_cast<unsigned>(p.A);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  int mismatch = 0;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int sum = 0, own = 0;
    for (int r = 0; r < N; ++r) {
      const int v = p.all_counts[static_cast<size_t>(r) * E + e];
      sum += v;
      if (r == rank) own = v;
    }
    if (own != mine[e]) mismatch = 1;
    tall[e] = sum;
  }
  mismatch = __syncthreads_or(mismatch);
  int ovf = 0;
  for (int q = warp; q < N; q += nwarps) {
    const int qlo = q * eloc, per = (eloc + 31) / 32;
    const int lo = qlo + min(lane * per, eloc), hi = qlo + min(lane * per + per, eloc);
    int sp = 0, sd = 0;
    for (int e = lo; e < hi; ++e) {
      const unsigned c = static_cast<unsigned>(tall[e]);
      const unsigned pe = roundup(c, A, p.a_log2);
      sp += static_cast<int>(pe);
      sd += static_cast<int>(pe - c);
    }
    int ip = sp, id = sd;
#pragma unroll 1
    for (int d = 1; d < 32; d <<= 1) {
      const int y = __shfl_up_sync(kFull, ip, d);
      const int z = __shfl_up_sync(kFull, id, d);
      if (lane >= d) {
        ip += y;
        id += z;
      }
    }
    int rp = ip - sp, rd = id - sd;
    for (int e = lo; e < hi; ++e) {
      const unsigned c = static_cast<unsigned>(tall[e]);
      const unsigned pe = roundup(c, A, p.a_log2);
      off_s[e] = rp;
      pad_s[e] = rd;
      rp += static_cast<int>(pe);
      rd += static_cast<int>(pe - c);
    }
    if (lane == 31) {
      if (static_cast<long long>(ip) > p.R) ovf = 1;
      if (q == rank) {
        off_s[E] = ip;  // this owner's P
        pad_s[E] = id;  // and its padding rows
      }
    }
  }
  ovf = __syncthreads_or(ovf);
  const int P = off_s[E], npad = pad_s[E], own_lo = rank * eloc;
  if (part == 0) {
    for (int j = threadIdx.x; j < eloc; j += blockDim.x) {
      p.counts[j] = tall[own_lo + j];
      p.counts_user[j] = tall[own_lo + j];
      p.offsets[j] = off_s[own_lo + j];
    }
    if (threadIdx.x == 0) {
      p.offsets[eloc] = P;
      unsigned st = bad ? EP_ST_BAD_INDEX : 0u;
      if (ovf) st |= EP_ST_OVERFLOW;
      if (mismatch) st |= EP_ST_COUNTS_MISMATCH;
      p.hdr[kHdrStatus] = static_cast<int>(st);
      p.hdr[kHdrT] = p.T;
      p.hdr[kHdrP] = P;
      p.hdr[kHdrNPad] = npad;
      p.hdr[kHdrA] = p.A;
      p.hdr[kHdrV] = P - npad;
      p.hdr[kHdrMagic] = kPreparedMagic;
    }
  }
  // This owner's padding rows, ascending, one warp per expert.
  if (npad > 0 && !ovf && !mismatch && npad <= p.pad_cap) {
    for (int j = part * nwarps + warp; j < eloc; j += nparts * nwarps) {
      const int e = own_lo + j;
      const unsigned c = static_cast<unsigned>(tall[e]);
      const int n = static_cast<int>(roundup(c, A, p.a_log2) - c);
      const int first = off_s[e] + static_cast<int>(c);
      for (int i = lane; i < n; i += 32) p.pad_list[pad_s[e] + i] = first + i;
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int before = 0;
    for (int r = 0; r < rank; ++r) before += p.all_counts[static_cast<size_t>(r) * E + e];
    off_s[e] += before;
  }
}

template <int MODE>
__global__ void __launch_bounds__(512, 1) ep_prepare_cluster_kernel(RouteParams p) {
  pdl_wait();
  pdl_trigger();
  cg::cluster_group cluster = cg::this_cluster();
  const int C = static_cast<int>(cluster.num_blocks());
  const int c = static_cast<int>(cluster.block_rank());
  extern __shared__ __align__(16) int smem[];
  const int W = blockDim.x >> 5, E = p.E, warp = threadIdx.x >> 5;
  int* wcnt = smem;              // [W][E]
  int* tot = wcnt + W * E;       // [E]  this CTA's totals, read by the whole cluster
  int* base = tot + E;           // [E]  routes to e in lower-ranked CTAs
  int* cnt_s = base + E;         // [E]
  int* off_s = cnt_s + E;        // [E+1]
  int* pad_s = off_s + E + 1;    // [E+1]
  int* flag_s = pad_s + E + 1;   // [1]  this CTA saw an index outside [-1, E)
  const int cbase = c * p.chunk, cend = min(cbase + p.chunk, p.n);
  const int per = p.chunk / W;
  const int lo = min(cbase + warp * per, cend), hi = min(lo + per, cend);
  int bad = 0;
  Packed pk;
  warp_load_count(p.idx, lo, hi, E, wcnt + warp * E, pk, bad);
  bad = __syncthreads_or(bad);
  column_prefix(wcnt, W, E, nullptr, nullptr, tot);  // relative to this CTA
  const int* counts = tot;
  if (C > 1) {
    if (threadIdx.x == 0) flag_s[0] = bad;
    cluster_arrive_release();
    cluster_wait();  // every CTA's totals and flag are visible to the cluster
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
      int b = 0, all = 0;
      for (int r = 0; r < C; ++r) {
        const int v = cluster.map_shared_rank(tot, r)[e];
        if (r < c) b += v;
        all += v;
      }
      base[e] = b;
      cnt_s[e] = all;
    }
    int remote_bad = 0;
    if (static_cast<int>(threadIdx.x) < C)
      remote_bad = *cluster.map_shared_rank(flag_s, static_cast<int>(threadIdx.x));
    bad = __syncthreads_or(remote_bad);
    // Done reading the other CTAs' shared memory; the matching wait comes at
    // the end, so that no CTA exits while another may still read from it.
    cluster_arrive_relaxed();
    counts = cnt_s;
  } else {
    __syncthreads();
  }
  if (MODE == kModeCount) {
    if (c == 0)
      for (int e = threadIdx.x; e < E; e += blockDim.x) p.counts_user[e] = counts[e];
    if (C > 1) cluster_wait();
    return;
  }
  if (MODE == kModeShard) {
    shard_finalize(p, counts, flag_s + 4, off_s, pad_s, bad, c, C);
  } else {
    int P = 0, npad = 0;
    finalize_compute(p, counts, off_s, pad_s, &P, &npad);
    finalize_write(p, counts, off_s, pad_s, P, npad, bad, c, C);
  }
  column_add(wcnt, W, E, off_s, C > 1 ? base : nullptr);
  __syncthreads();
  if (MODE == kModeShard)
    warp_assign(pk, lo, hi, E, wcnt + warp * E, p.slot, p.dest, E / p.nranks);
  else
    warp_assign(pk, lo, hi, E, wcnt + warp * E, p.slot);
  if (C > 1) cluster_wait();
}

// ---------------------------------------------------------------------------
// Grid-wide routing map: one cooperative launch of G CTAs (all resident at
// once), each counting and assigning a chunk of routes, with one grid-wide
// wait between counting and assigning.  For batches whose slot assignment
// would keep a 16-CTA cluster's SMs busy: assignment is bound by instruction
// issue per SM, and G CTAs spread it over G SMs.
// ---------------------------------------------------------------------------

// Waits until every CTA of the grid has arrived, on one arrival word that
// returns to its starting value after each wait: CTA 0 adds 2^31 - (G - 1),
// every other CTA adds 1, so the G arrivals together add exactly 2^31 and
// flip the word's top bit, which each CTA waits to see change from the value
// its own addition returned.  Bounded: false after kBarrierSpins polls (about
// a second) for the caller to give up.  Every thread's earlier global writes
// are visible to every CTA afterwards.
constexpr unsigned kBarrierSpins = 1u << 20;

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ bool grid_barrier(unsigned* word) {
  __shared__ int ok_s;
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned add = blockIdx.x == 0 ? 0x80000000u - (gridDim.x - 1u) : 1u;
    __threadfence();
    const unsigned old = atomicAdd(word, add);
    int ok = 1;
    unsigned spins = 0;
    while (((ld_acquire_gpu(word) ^ old) & 0x80000000u) == 0u) {
      if (++spins > kBarrierSpins) {
        ok = 0;
        break;
      }
      __nanosleep(32);
    }
    __threadfence();
    ok_s = ok;
  }
  __syncthreads();
  return ok_s != 0;
}

// Phases: (1) count the chunk per warp, per-warp bases inside the chunk,
// publish the chunk's per-expert totals (one row of hist per chunk, rows of
// E rounded up to 4 words) and its invalid-index flag; wait for the grid.
// (2) Every CTA reads all rows: the totals over all chunks, and the routes to
// each expert in the chunks before its own.  (3) Every CTA computes the
// aligned offsets (CTA 0 writes counts, offsets and header, every CTA a share
// of the padding list) and assigns the slots of its chunk.
__global__ void __launch_bounds__(512, 1) ep_prepare_wide_kernel(RouteParams p) {
  pdl_wait();
  pdl_trigger();
  // After a wait gave up the arrival word is not known to be consistent:
  // the handle stays refused until its memory is zero-filled.
  if (__ldcg(p.hdr + kHdrMagic) == kTimedOutMagic) return;
  extern __shared__ __align__(16) int smem[];
  const int G = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
  const int W = blockDim.x >> 5, E = p.E, warp = threadIdx.x >> 5;
  const int Es = (E + 3) & ~3;
  int* wcnt = smem;              // [W][E]
  int* tot = wcnt + W * E;       // [E] this chunk's totals, then its bases
  int* cnt_s = tot + E;          // [E] totals over all chunks
  int* off_s = cnt_s + E;        // [E+1]
  int* pad_s = off_s + E + 1;    // [E+1]
  const int cbase = c * p.chunk, cend = min(cbase + p.chunk, p.n);
  const int per = p.chunk / W;
  const int lo = min(cbase + warp * per, cend), hi = min(lo + per, cend);
  int bad = 0;
  Packed pk;
  warp_load_count(p.idx, lo, hi, E, wcnt + warp * E, pk, bad);
  bad = __syncthreads_or(bad);
  column_prefix(wcnt, W, E, nullptr, nullptr, tot);
  int* hrow = p.hist + static_cast<size_t>(c) * Es;
  for (int e = threadIdx.x; e < E; e += blockDim.x) hrow[e] = tot[e];
  if (threadIdx.x == 0) p.badflag[c] = bad;
  if (!grid_barrier(reinterpret_cast<unsigned*>(p.hdr + kHdrBarrier))) {
    if (threadIdx.x == 0) atomicExch(p.hdr + kHdrMagic, kTimedOutMagic);
    return;
  }
  // (2) S consecutive lanes share 4 experts (one 16-byte column of hist) and
  // split the rows among them; shuffles add up the S partial sums.
  {
    const int Q = Es >> 2;
    int S = 1;
    while (S < 32 && Q * S * 2 <= static_cast<int>(blockDim.x)) S <<= 1;
    const int sub = threadIdx.x & (S - 1), per_pass = blockDim.x / S;
#pragma unroll 1
    for (int q0 = 0; q0 < Q; q0 += per_pass) {
      const int q = q0 + static_cast<int>(threadIdx.x) / S;
      int4 all = make_int4(0, 0, 0, 0), below = make_int4(0, 0, 0, 0);
      if (q < Q) {
        const int4* col = reinterpret_cast<const int4*>(p.hist) + q;
#pragma unroll 4
        for (int g = sub; g < G; g += S) {
          const int4 v = __ldcg(col + static_cast<size_t>(g) * Q);
          all.x += v.x; all.y += v.y; all.z += v.z; all.w += v.w;
          if (g < c) {
            below.x += v.x; below.y += v.y; below.z += v.z; below.w += v.w;
          }
        }
      }
#pragma unroll 1
      for (int d = 1; d < S; d <<= 1) {
        all.x += __shfl_xor_sync(kFull, all.x, d);
        all.y += __shfl_xor_sync(kFull, all.y, d);
        all.z += __shfl_xor_sync(kFull, all.z, d);
        all.w += __shfl_xor_sync(kFull, all.w, d);
        below.x += __shfl_xor_sync(kFull, below.x, d);
        below.y += __shfl_xor_sync(kFull, below.y, d);
        below.z += __shfl_xor_sync(kFull, below.z, d);
        below.w += __shfl_xor_sync(kFull, below.w, d);
      }
      if (q < Q && sub == 0) {
        const int e = 4 * q;
        const int av[4] = {all.x, all.y, all.z, all.w}, bv[4] = {below.x, below.y, below.z, below.w};
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (e + j < E) {
            cnt_s[e + j] = av[j];
            tot[e + j] = bv[j];
          }
      }
    }
  }
  if (c == 0) {
    int b = 0;
    for (int g = threadIdx.x; g < G; g += blockDim.x) b |= __ldcg(p.badflag + g);
    bad = b;
  }
  bad = __syncthreads_or(bad);
  // (3)
  int P = 0, npad = 0;
  finalize_compute(p, cnt_s, off_s, pad_s, &P, &npad);
  finalize_write(p, cnt_s, off_s, pad_s, P, npad, bad, c, G);
  column_add(wcnt, W, E, off_s, tot);
  __syncthreads();
  warp_assign(pk, lo, hi, E, wcnt + warp * E, p.slot);
}

// Shared set-up of the chunked kernels: load the chunk, count per warp.
struct ChunkCtx {
  int* wcnt;
  int lo, hi, bad;
};

__device__ __forceinline__ ChunkCtx chunk_count(const RouteParams& p, int* smem, Packed& pk) {
  ChunkCtx c;
  const int W = blockDim.x >> 5, E = p.E, warp = threadIdx.x >> 5;
  c.wcnt = smem;
  const int cbase = blockIdx.x * p.chunk;
  const int cend = min(cbase + p.chunk, p.n);
  const int per = p.chunk / W;
  c.lo = min(cbase + warp * per, cend);
  c.hi = min(c.lo + per, cend);
  c.bad = 0;
  warp_load_count(p.idx, c.lo, c.hi, E, c.wcnt + warp * E, pk, c.bad);
  c.bad = __syncthreads_or(c.bad);
  return c;
}

__global__ void __launch_bounds__(512) ep_route_hist_kernel(RouteParams p) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ __align__(16) int smem[];
  Packed pk;
  const ChunkCtx c = chunk_count(p, smem, pk);
  const int W = blockDim.x >> 5, E = p.E;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int s = 0;
    for (int w = 0; w < W; ++w) s += c.wcnt[w * E + e];
    p.hist[static_cast<size_t>(blockIdx.x) * E + e] = s;
  }
  if (threadIdx.x == 0) p.badflag[blockIdx.x] = c.bad;
  if (blockIdx.x == 0 && threadIdx.x == 0) p.hdr[kHdrTicket] = 0;  // for the scan kernel
}

// The scan kernel: kScanWarps experts per CTA, ceil(E / kScanWarps) CTAs.
// Shared memory (the last CTA only), ints: counts [E], offsets and padding
// scans [E+1] each.
constexpr int kScanWarps = 8;
__host__ __device__ constexpr size_t scan_kernel_smem_bytes(int E) {
  return static_cast<size_t>(3 * E + 2) * 4;
}

// Exclusive scan over chunks per expert, in place: hist[c][e] becomes the
// number of routes to e in chunks before c, and counts[e] the total.  One
// warp per expert; lane q owns the contiguous run of chunks [q*L, q*L + L)
// (held in registers between the two passes when L <= 8, i.e. up to 256
// chunks), and a shuffle scan of the run sums gives each run its base.  Then
// each CTA takes a ticket; the last one to finish (its writers fenced before
// their tickets) reads the totals and computes the aligned offsets, the
// header and the padding list.  No CTA waits for another.
__global__ void __launch_bounds__(kScanWarps * 32) ep_route_scan_kernel(RouteParams p) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ __align__(16) int smem[];
  __shared__ int last_s;
  const int E = p.E, NC = p.nchunks, lane = threadIdx.x & 31;
  const int e = blockIdx.x * kScanWarps + static_cast<int>(threadIdx.x >> 5);
  if (e < E) {
    const int L = (NC + 31) / 32;
    const int c0 = min(NC, lane * L), c1 = min(NC, c0 + L);
    int* col = p.hist + e;  // hist[c][e] = col[c * E]
    int v[8];
    int sum = 0;
    if (L <= 8) {
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = c0 + j < c1 ? col[static_cast<size_t>(c0 + j) * E] : 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) sum += v[j];
    } else {
      for (int cb = c0; cb < c1; cb += 8) {
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = cb + j < c1 ? col[static_cast<size_t>(cb + j) * E] : 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) sum += v[j];
      }
    }
    int incl = sum;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int y = __shfl_up_sync(kFull, incl, d);
      if (lane >= d) incl += y;
    }
    const int total = __shfl_sync(kFull, incl, 31);
    int run = incl - sum;
    if (L <= 8) {
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (c0 + j < c1) {
          col[static_cast<size_t>(c0 + j) * E] = run;
          run += v[j];
        }
    } else {
      for (int cb = c0; cb < c1; cb += 8) {
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = cb + j < c1 ? col[static_cast<size_t>(cb + j) * E] : 0;
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (cb + j < c1) {
            col[static_cast<size_t>(cb + j) * E] = run;
            run += v[j];
          }
      }
    }
    if (lane == 0) p.counts[e] = total;
  }
  __threadfence();  // this CTA's totals are visible before its ticket
  __syncthreads();
  if (threadIdx.x == 0) last_s = atomicAdd(p.hdr + kHdrTicket, 1) == static_cast<int>(gridDim.x) - 1;
  __syncthreads();
  if (!last_s) return;
  __threadfence();
  int* cnt_s = smem;           // [E]
  int* off_s = cnt_s + E;      // [E+1]
  int* pad_s = off_s + E + 1;  // [E+1]
  for (int i = threadIdx.x; i < E; i += blockDim.x) cnt_s[i] = __ldcg(p.counts + i);
  int bad = 0;
  for (int c = threadIdx.x; c < NC; c += blockDim.x) bad |= __ldcg(p.badflag + c);
  bad = __syncthreads_or(bad);
  int P = 0, npad = 0;
  finalize_compute(p, cnt_s, off_s, pad_s, &P, &npad);
  finalize_write(p, cnt_s, off_s, pad_s, P, npad, bad, 0, 1);
  if (threadIdx.x == 0) p.hdr[kHdrTicket] = 0;
}

__global__ void __launch_bounds__(512) ep_route_assign_kernel(RouteParams p) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ __align__(16) int smem[];
  const int W = blockDim.x >> 5, E = p.E;
  // This chunk's base row per expert (offset + routes in earlier chunks),
  // loaded before the recount so that the two latencies overlap.
  int* base_s = smem + W * E;  // [E]
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    base_s[e] = __ldg(p.offsets + e) + p.hist[static_cast<size_t>(blockIdx.x) * E + e];
  Packed pk;
  const ChunkCtx c = chunk_count(p, smem, pk);  // syncs: base_s is visible after it
  column_prefix(c.wcnt, W, E, base_s, nullptr, nullptr);
  __syncthreads();
  warp_assign(pk, c.lo, c.hi, E, c.wcnt + (threadIdx.x >> 5) * E, p.slot);
}

// Rank-major layers: per route, the owner rank of its expert where this is
// the owner's first route in the token (the route the row goes with), -1 at
// the token's other routes to that owner and at masked routes, and nranks
// for an index outside [-1, E) (the routing map then flags and masks it);
// beside it every valid route's owner.  One thread per token, its K <= KMAX
// indices loaded together before the serial pass over them.
template <int KMAX>
__global__ void __launch_bounds__(256) ep_rank_major_owners_kernel(RouteParams p) {
  pdl_wait();
  pdl_trigger();
  const int K = p.K;
  const int stride = static_cast<int>(gridDim.x * blockDim.x);
  for (int t = static_cast<int>(blockIdx.x * blockDim.x + threadIdx.x); t < p.T; t += stride) {
    const long long* in = p.idx_in + static_cast<size_t>(t) * K;
    long long e[KMAX];
#pragma unroll
    for (int k = 0; k < KMAX; ++k) e[k] = k < K ? __ldg(in + k) : -1LL;
    unsigned long long seen = 0ull;
#pragma unroll
    for (int k = 0; k < KMAX; ++k) {
      if (k >= K) break;
      long long o = -1;
      int own = -1;
      if (e[k] >= 0 && e[k] < p.E_all) {
        own = static_cast<int>(e[k] / p.eloc);
        if (((seen >> own) & 1ull) == 0ull) {
          o = own;
          seen |= 1ull << own;
        }
      } else if (e[k] != -1) {
        o = p.nranks;
      }
      const size_t i = static_cast<size_t>(t) * K + k;
      p.oidx[i] = o;
      p.owner[i] = own;
    }
  }
}

}  // namespace

int cluster_warps(int E) {
  int w = kMaxW;
  while (w > 1 && cluster_smem_bytes(w, E) > static_cast<size_t>(kSmemBudget) - 1024) --w;
  return w;
}

int chunk_warps(int E) {
  return std::max(1, std::min(kChunkWarpsMax, 32768 / (4 * E)));
}

// Fails when this device cannot run the sm_103a image.
cudaError_t probe_kernel_image() {
  cudaFuncAttributes a;
  return cudaFuncGetAttributes(&a, ep_prepare_cluster_kernel<kModeLocal>);
}

bool prepare_is_one_launch(long long n, int E, int max_cluster) {
  return n <= static_cast<long long>(max_cluster) * cluster_warps(E) * 32 * kMaxJ;
}

int prepare_max_cluster() {
  if (cudaFuncSetAttribute(ep_prepare_cluster_kernel<kModeLocal>, cudaFuncAttributeNonPortableClusterSizeAllowed,
                           1) != cudaSuccess) {
    cudaGetLastError();
    return kMaxCluster;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kMaxClusterWide);
  cfg.blockDim = dim3(kChunkWarpsMax * 32);
  cfg.dynamicSmemBytes = static_cast<size_t>(kSmemBudget) - 1024;  // the most the kernel takes
  cudaLaunchAttribute at;
  at.id = cudaLaunchAttributeClusterDimension;
  at.val.clusterDim.x = kMaxClusterWide;
  at.val.clusterDim.y = 1;
  at.val.clusterDim.z = 1;
  cfg.attrs = &at;
  cfg.numAttrs = 1;
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, ep_prepare_cluster_kernel<kModeLocal>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return kMaxCluster;
  }
  return clusters >= 1 ? kMaxClusterWide : kMaxCluster;
}

// Shared memory of the grid-wide kernel: the cluster kernel's layout.
size_t wide_smem_bytes(int W, int E) { return cluster_smem_bytes(W, E); }

int prepare_wide_ctas() {
  int dev = 0, sms = 0, coop = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess || !coop) {
    cudaGetLastError();
    return 0;
  }
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, ep_prepare_wide_kernel, kMaxW * 32,
                                                    static_cast<size_t>(kSmemBudget) - 1024) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return per_sm * sms;
}

// Routes above which prepare runs grid-wide (when the device allows it): at
// and below, the cluster's few SMs assign slots as fast as the grid-wide
// kernel's wait and table read cost (65,536 routes at 128 experts: 12.3 us
// both ways; 131,072 at 256 experts: 16.6 us in the cluster, 14.3 us
// grid-wide, on a GB300).
constexpr long long kWideMinRoutes = 65536;
// Routes per warp the grid-wide kernel's CTA count is chosen for (64 made
// every CTA read twice the table for no faster assignment).
constexpr long long kWideRoutesPerWarp = 128;
// Words of the chunk-total table every CTA of the grid-wide kernel reads.
constexpr long long kWideMaxTableWords = 65536;

cudaError_t launch_prepare(const RouteParams& p0, int num_sms, int max_cluster, int wide_ctas,
                           cudaStream_t s, int* launches) {
  RouteParams p = p0;
  *launches = 0;
  const int Wc = cluster_warps(p.E);
  // Grid-wide: up to one CTA per SM, sized for kWideRoutesPerWarp, at most
  // the hist rows of the handle (p.nchunks), the CTAs that fit at once and
  // a table of kWideMaxTableWords.
  if (p.n > kWideMinRoutes && wide_ctas > 0) {
    const long long Es = (p.E + 3) & ~3;
    const long long gmax = std::min<long long>(std::min<long long>(std::min<long long>(wide_ctas, num_sms), p.nchunks),
                                               kWideMaxTableWords / Es);
    const long long want = (p.n + static_cast<long long>(Wc) * kWideRoutesPerWarp - 1) /
                           (static_cast<long long>(Wc) * kWideRoutesPerWarp);
    const long long G0 = std::max<long long>(1, std::min(gmax, want));
    long long rpw = (p.n + G0 * Wc - 1) / (G0 * Wc);
    rpw = std::max<long long>(32, ((rpw + 31) / 32) * 32);
    if (rpw <= 32 * kMaxJ) {
      RouteParams q = p;
      q.warps = Wc;
      q.chunk = static_cast<int>(rpw * Wc);
      const int G = static_cast<int>((q.n + q.chunk - 1) / q.chunk);  // <= G0
      q.nchunks = G;
      const cudaError_t e = launch_pdl_ex(ep_prepare_wide_kernel, dim3(G), dim3(Wc * 32),
                                          wide_smem_bytes(Wc, q.E), s, 0u, true, q);
      if (e != cudaErrorCooperativeLaunchTooLarge) {
        *launches = e == cudaSuccess ? 1 : 0;
        return e;
      }
      // Refused because the CTAs cannot all be resident here (a context
      // limited to part of the GPU): a launch error that does not stick.
      // Clear it and take the cluster or chunked path below.
      cudaGetLastError();
    }
  }
  if (prepare_is_one_launch(p.n, p.E, max_cluster)) {
    // One cluster launch.  Assigning slots is instruction-bound, so the CTA
    // count is picked for kClusterRoutesPerWarp routes per warp; with all
    // max_cluster CTAs in use, up to 512 routes per warp a single launch
    // still beat the three chunked kernels (8 CTAs, Qwen3-sized batch: 15.2
    // against 17.6 us; 16 CTAs: Qwen3 12.3 us, DeepSeek-V3 16.8 against
    // 22.3 us); beyond it the chunked kernels spread the work over many SMs.
    const long long per_cta = static_cast<long long>(Wc) * kClusterRoutesPerWarp;
    int C = static_cast<int>(std::min<long long>(max_cluster, std::max<long long>(1, (p.n + per_cta - 1) / per_cta)));
    long long rpw = (p.n + static_cast<long long>(C) * Wc - 1) / (static_cast<long long>(C) * Wc);
    rpw = std::max<long long>(32, ((rpw + 31) / 32) * 32);
    p.warps = Wc;
    p.chunk = static_cast<int>(rpw * Wc);
    C = static_cast<int>(std::max<long long>(1, (p.n + p.chunk - 1) / p.chunk));
    p.nchunks = C;
    *launches = 1;
    return launch_pdl(ep_prepare_cluster_kernel<kModeLocal>, dim3(C), dim3(Wc * 32), cluster_smem_bytes(Wc, p.E),
                      s, static_cast<unsigned>(C), p);
  }
  // p.nchunks arrives as the capacity of hist (chunks); pick routes per warp
  // (a multiple of 32, at most the 32*kMaxJ a warp holds) for about one CTA
  // per SM, more chunks when the routes need them, never more than the
  // capacity (registration guarantees 32*kMaxJ routes per warp suffice).
  const int W = chunk_warps(p.E);
  const long long cap = p.nchunks;
  const long long target = std::min<long long>(cap, static_cast<long long>(num_sms));
  long long rpw = (p.n + target * W - 1) / (target * W);
  rpw = std::min<long long>(32 * kMaxJ, std::max<long long>(32, ((rpw + 31) / 32) * 32));
  while ((p.n + rpw * W - 1) / (rpw * W) > cap && rpw < 32 * kMaxJ) rpw += 32;
  if ((p.n + rpw * W - 1) / (rpw * W) > cap) return cudaErrorInvalidConfiguration;
  p.warps = W;
  p.chunk = static_cast<int>(rpw * W);
  p.nchunks = static_cast<int>((p.n + p.chunk - 1) / p.chunk);
  const size_t chunk_smem = static_cast<size_t>(W) * p.E * 4;
  const size_t assign_smem = static_cast<size_t>(W + 1) * p.E * 4;
  const size_t scan_smem = scan_kernel_smem_bytes(p.E);
  cudaError_t e = launch_pdl(ep_route_hist_kernel, dim3(p.nchunks), dim3(W * 32), chunk_smem, s, 0u, p);
  if (e != cudaSuccess) return e;
  const unsigned scan_ctas = static_cast<unsigned>((p.E + kScanWarps - 1) / kScanWarps);
  e = launch_pdl(ep_route_scan_kernel, dim3(scan_ctas), dim3(kScanWarps * 32), scan_smem, s, 0u, p);
  if (e != cudaSuccess) return e;
  e = launch_pdl(ep_route_assign_kernel, dim3(p.nchunks), dim3(W * 32), assign_smem, s, 0u, p);
  *launches = 3;
  return e;
}

// ---------------------------------------------------------------------------
// Sharded layers: the count-only and sharded modes of the cluster kernel, on
// a cluster of up to 16 CTAs where the device runs one (shard_max_cluster),
// else kMaxCluster.
// ---------------------------------------------------------------------------
namespace {
int shard_warps(int E) {
  int w = kMaxW;
  while (w > 1 && cluster_smem_bytes(w, E, true) > static_cast<size_t>(kSmemBudget) - 1024) --w;
  return w;
}

cudaError_t launch_cluster_mode(const RouteParams& p0, bool count_only, int max_cluster,
                                cudaStream_t s) {
  RouteParams p = p0;
  const int Wc = shard_warps(p.E);
  const long long per_cta = static_cast<long long>(Wc) * kClusterRoutesPerWarp;
  int C = static_cast<int>(std::min<long long>(max_cluster, std::max<long long>(1, (p.n + per_cta - 1) / per_cta)));
  long long rpw = (p.n + static_cast<long long>(C) * Wc - 1) / (static_cast<long long>(C) * Wc);
  rpw = std::max<long long>(32, ((rpw + 31) / 32) * 32);
  if (rpw > 32 * kMaxJ) return cudaErrorInvalidConfiguration;  // registration keeps n below this
  p.warps = Wc;
  p.chunk = static_cast<int>(rpw * Wc);
  C = static_cast<int>(std::max<long long>(1, (p.n + p.chunk - 1) / p.chunk));
  p.nchunks = C;
  const size_t smem = cluster_smem_bytes(Wc, p.E, true);
  if (count_only)
    return launch_pdl(ep_prepare_cluster_kernel<kModeCount>, dim3(C), dim3(Wc * 32), smem, s,
                      static_cast<unsigned>(C), p);
  return launch_pdl(ep_prepare_cluster_kernel<kModeShard>, dim3(C), dim3(Wc * 32), smem, s,
                    static_cast<unsigned>(C), p);
}
}  // namespace

long long shard_max_routes(int E, int max_cluster) {
  return static_cast<long long>(max_cluster) * shard_warps(E) * 32 * kMaxJ;
}

// Largest cluster of the count and sharded modes on the current device: 16
// CTAs when one such cluster of the sharded instance fits (the non-portable
// size is allowed on both instances here), else kMaxCluster.
int shard_max_cluster() {
  if (cudaFuncSetAttribute(ep_prepare_cluster_kernel<kModeCount>,
                           cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess ||
      cudaFuncSetAttribute(ep_prepare_cluster_kernel<kModeShard>,
                           cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
    cudaGetLastError();
    return kMaxCluster;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kMaxClusterWide);
  cfg.blockDim = dim3(kChunkWarpsMax * 32);
  cfg.dynamicSmemBytes = static_cast<size_t>(kSmemBudget) - 1024;  // the most the kernel takes
  cudaLaunchAttribute at;
  at.id = cudaLaunchAttributeClusterDimension;
  at.val.clusterDim.x = kMaxClusterWide;
  at.val.clusterDim.y = 1;
  at.val.clusterDim.z = 1;
  cfg.attrs = &at;
  cfg.numAttrs = 1;
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, ep_prepare_cluster_kernel<kModeShard>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return kMaxCluster;
  }
  return clusters >= 1 ? kMaxClusterWide : kMaxCluster;
}

cudaError_t launch_shard_count(const RouteParams& p, int max_cluster, cudaStream_t s, int* launches) {
  *launches = 1;
  return launch_cluster_mode(p, true, max_cluster, s);
}

cudaError_t launch_shard_prepare(const RouteParams& p, int max_cluster, cudaStream_t s,
                                 int* launches) {
  *launches = 1;
  return launch_cluster_mode(p, false, max_cluster, s);
}

// ---------------------------------------------------------------------------
// Routing map with the per-chunk counters in a fixed device array, for
// callers that cannot allocate device memory (ep_prepare_static_scratch).
//
// The array lives in every GPU that loads this library, for the life of the
// process.  Every call reuses it and it keeps the last call's contents.
// Nothing in it has to start at zero: the histogram kernel writes every
// counter and flag that the scan and assign kernels later read.  Two calls
// that run on the GPU at the same time (two streams, or two handles without
// ordering between them) overwrite each other's counters and race.
// ---------------------------------------------------------------------------
static __device__ __align__(256) int g_prepare_scratch[kStaticScratchInts];

namespace {
std::mutex g_scratch_mu;
int* g_scratch_ptr[64] = {};
}  // namespace

// Device address of g_prepare_scratch on the current device, looked up once
// per device (the host-side name of a __device__ array is not a device
// address).  This lookup is what the first call on a device does, which is
// why that first call belongs before any stream capture.
cudaError_t static_scratch_address(int** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_prepare_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = static_cast<int*>(ptr);
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

// Chunk plan for the fixed array: (E + 1) * chunks counters must fit in it.
// Routes per warp aim at about two chunks per SM, are capped at the 32*kMaxJ
// a warp holds in registers, and only then is the chunk count allowed to grow
// past that aim; it may grow up to what the array holds.  Returns false only
// when even chunks of 32*kMaxJ routes per warp need more counters than the
// array has (the caller reports EP_ERR_LIMIT).
bool static_scratch_plan(int n, int E, int num_sms, int* warps, int* chunk, int* nchunks) {
  const int W = chunk_warps(E);
  const long long cap = kStaticScratchInts / (E + 1);
  if (cap < 1) return false;
  const long long target = std::max(1LL, std::min<long long>(cap, 2LL * num_sms));
  long long rpw = (n + target * W - 1) / (target * W);
  rpw = std::min<long long>(32 * kMaxJ, std::max<long long>(32, ((rpw + 31) / 32) * 32));
  const long long ch = rpw * W;
  const long long nch = std::max(1LL, (n + ch - 1) / ch);
  if (nch > cap) return false;
  *warps = W;
  *chunk = static_cast<int>(ch);
  *nchunks = static_cast<int>(nch);
  return true;
}

cudaError_t launch_prepare_static_scratch(const RouteParams& p0, int* scratch, int num_sms,
                                          cudaStream_t s, int* launches) {
  RouteParams p = p0;
  *launches = 0;
  if (!static_scratch_plan(p.n, p.E, num_sms, &p.warps, &p.chunk, &p.nchunks))
    return cudaErrorInvalidValue;
  p.hist = scratch;
  p.badflag = scratch + static_cast<size_t>(p.E) * p.nchunks;
  const int W = p.warps;
  const size_t chunk_smem = static_cast<size_t>(W) * p.E * 4;
  const size_t assign_smem = static_cast<size_t>(W + 1) * p.E * 4;
  const size_t scan_smem = scan_kernel_smem_bytes(p.E);
  ep_route_hist_kernel<<<p.nchunks, W * 32, chunk_smem, s>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  ep_route_scan_kernel<<<(p.E + kScanWarps - 1) / kScanWarps, kScanWarps * 32, scan_smem, s>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  ep_route_assign_kernel<<<p.nchunks, W * 32, assign_smem, s>>>(p);
  *launches = 3;
  return cudaGetLastError();
}

cudaError_t launch_rank_major_owners(const RouteParams& p, int num_sms, cudaStream_t s) {
  const long long want = (static_cast<long long>(p.T) + 255) / 256;
  const dim3 grid(static_cast<unsigned>(std::max(1LL, std::min(want, static_cast<long long>(num_sms) * 8))));
  if (p.K <= 2) return launch_pdl(ep_rank_major_owners_kernel<2>, grid, dim3(256), 0, s, 0u, p);
  if (p.K <= 4) return launch_pdl(ep_rank_major_owners_kernel<4>, grid, dim3(256), 0, s, 0u, p);
  if (p.K <= 8) return launch_pdl(ep_rank_major_owners_kernel<8>, grid, dim3(256), 0, s, 0u, p);
  if (p.K <= 16) return launch_pdl(ep_rank_major_owners_kernel<16>, grid, dim3(256), 0, s, 0u, p);
  return launch_pdl(ep_rank_major_owners_kernel<32>, grid, dim3(256), 0, s, 0u, p);
}

}  // namespace ep
