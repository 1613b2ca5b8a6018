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
// lane part comes from __match_any_sync (lanes holding the same expert) and a
// population count of the lower lanes; the warp part from per-warp counters in
// shared memory; the chunk part from an exclusive scan over chunks.  No atomics
// decide an order, so every slot is the unique stable one.
//
// Two shapes:
//   cluster: one launch of a thread-block cluster of up to 8 CTAs.  Each CTA
//            counts its chunk, the CTAs read each other's per-expert totals
//            through distributed shared memory, each computes the aligned
//            offsets, and each assigns the slots of its chunk (decode to
//            DeepSeek-V3-sized batches);
//   chunked: ep_route_hist (per-chunk counts) -> ep_route_scan (one CTA: scan
//            over chunks per expert, aligned scan over experts, padding list)
//            -> ep_route_assign (slots), for batches beyond the cluster's reach
//            and for the fixed-scratch entry point.
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

// Expert ids of routes [lo, hi) into the shared cache (index r - cbase).
__device__ __forceinline__ void warp_load(const long long* __restrict__ idx, int lo, int hi,
                                          int cbase, int E, short* ecache, int& bad) {
  const int lane = threadIdx.x & 31;
#pragma unroll 4
  for (int r = lo + lane; r < hi; r += 32)
    ecache[r - cbase] = static_cast<short>(decode_expert(__ldg(idx + r), E, bad));
  __syncwarp();
}

// Adds this warp's route counts per expert to its own counter row.
__device__ __forceinline__ void warp_count(int lo, int hi, int cbase, const short* ecache,
                                           int* wrow) {
  const int lane = threadIdx.x & 31;
  for (int base = lo; base < hi; base += 32) {
    const int r = base + lane;
    const int e = r < hi ? ecache[r - cbase] : -1;
    const unsigned m = __match_any_sync(kFull, e);
    if (e >= 0 && lane == __ffs(m) - 1) wrow[e] += __popc(m);
    __syncwarp();
  }
}

// Slots of this warp's routes; wbase[e] is the next free row of expert e for
// this warp and advances as routes are placed.
__device__ __forceinline__ void warp_assign(int lo, int hi, int cbase, const short* ecache,
                                            int* wbase, int* __restrict__ slot) {
  const int lane = threadIdx.x & 31;
  const unsigned lower = (1u << lane) - 1u;
  for (int base = lo; base < hi; base += 32) {
    const int r = base + lane;
    const int e = r < hi ? ecache[r - cbase] : -1;
    const unsigned m = __match_any_sync(kFull, e);
    int s = -1;
    if (e >= 0) s = wbase[e] + __popc(m & lower);
    __syncwarp();
    if (e >= 0 && lane == __ffs(m) - 1) wbase[e] += __popc(m);
    __syncwarp();
    if (r < hi) slot[r] = s;
  }
}

// In-place exclusive scan of data[0, n) in shared memory by the whole CTA
// (blockDim.x a multiple of 32); returns the total.
__device__ int block_exclusive_scan(int* data, int n) {
  __shared__ int wsum[32];
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int nw = blockDim.x >> 5;
  const int per = (n + blockDim.x - 1) / blockDim.x;
  const int lo = min(tid * per, n), hi = min(lo + per, n);
  int local = 0;
  for (int i = lo; i < hi; ++i) local += data[i];
  int x = local;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int y = __shfl_up_sync(kFull, x, d);
    if (lane >= d) x += y;
  }
  if (lane == 31) wsum[w] = x;
  __syncthreads();
  if (w == 0) {
    int v = lane < nw ? wsum[lane] : 0;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int y = __shfl_up_sync(kFull, v, d);
      if (lane >= d) v += y;
    }
    if (lane < nw) wsum[lane] = v;
  }
  __syncthreads();
  int run = x - local + (w > 0 ? wsum[w - 1] : 0);
  const int total = wsum[nw - 1];
  for (int i = lo; i < hi; ++i) {
    const int t = data[i];
    data[i] = run;
    run += t;
  }
  __syncthreads();
  return total;
}

// Given c_e in cnt_s: off_s <- off_e (and off_s[E] = P), pad_s <- the
// exclusive scan of the padding rows per expert (pad_s[E] = their number).
// off_s and pad_s are [E+1] shared scratch.  Whole CTA.
__device__ void finalize_compute(const RouteParams& p, const int* cnt_s, int* off_s, int* pad_s,
                                 int* P_out, int* npad_out) {
  const int E = p.E, A = p.A;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int c = cnt_s[e];
    const int pe = ((c + A - 1) / A) * A;
    off_s[e] = pe;
    pad_s[e] = pe - c;
  }
  __syncthreads();
  const int P = block_exclusive_scan(off_s, E);
  const int npad = block_exclusive_scan(pad_s, E);
  if (threadIdx.x == 0) {
    off_s[E] = P;
    pad_s[E] = npad;
  }
  __syncthreads();
  *P_out = P;
  *npad_out = npad;
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
  // Padding rows, ascending: entry i belongs to the last expert e with
  // pad_s[e] <= i, and is its (i - pad_s[e])-th padding row.  Skipped when P
  // exceeds the capacity (the row calls then write nothing); otherwise
  // npad <= min(P, E*(A-1)) fits the list.
  const int nwrite = (static_cast<long long>(P) > p.R || npad > p.pad_cap) ? 0 : npad;
  for (int i = part * blockDim.x + threadIdx.x; i < nwrite; i += nparts * blockDim.x) {
    int lo = 0, hi = E - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (pad_s[mid] <= i) lo = mid; else hi = mid - 1;
    }
    p.pad_list[i] = off_s[lo] + cnt_s[lo] + (i - pad_s[lo]);
  }
}

__device__ void finalize(const RouteParams& p, const int* cnt_s, int* off_s, int* pad_s,
                         int bad) {
  int P = 0, npad = 0;
  finalize_compute(p, cnt_s, off_s, pad_s, &P, &npad);
  finalize_write(p, cnt_s, off_s, pad_s, P, npad, bad, 0, 1);
}

// Shared memory of the cluster kernel, in ints: per-warp counters [W][E],
// this CTA's totals [E], earlier CTAs' totals [E], counts [E], offsets and
// padding scans [E+1] each, a flag word (+3 pad), then W pieces of kPiece
// int16 expert ids.
__host__ __device__ constexpr size_t cluster_smem_bytes(int W, int E) {
  return static_cast<size_t>(W * E + 3 * E + 2 * (E + 1) + 4) * 4 +
         static_cast<size_t>(W) * kPiece * 2;
}

__global__ void __launch_bounds__(1024) ep_prepare_cluster_kernel(RouteParams p) {
  pdl_wait();
  pdl_trigger();
  cg::cluster_group cluster = cg::this_cluster();
  const int C = static_cast<int>(cluster.num_blocks());
  const int c = static_cast<int>(cluster.block_rank());
  extern __shared__ int smem[];
  const int W = blockDim.x >> 5, E = p.E, warp = threadIdx.x >> 5;
  int* wcnt = smem;              // [W][E]
  int* tot = wcnt + W * E;       // [E]  this CTA's totals, read by the whole cluster
  int* base = tot + E;           // [E]  routes to e in lower-ranked CTAs
  int* cnt_s = base + E;         // [E]
  int* off_s = cnt_s + E;        // [E+1]
  int* pad_s = off_s + E + 1;    // [E+1]
  int* flag_s = pad_s + E + 1;   // [1]  this CTA saw an index outside [-1, E)
  short* cache = reinterpret_cast<short*>(flag_s + 4) + warp * kPiece;
  for (int i = threadIdx.x; i < W * E; i += blockDim.x) wcnt[i] = 0;
  const int cbase = c * p.chunk, cend = min(cbase + p.chunk, p.n);
  const int per = p.chunk / W;
  const int lo = min(cbase + warp * per, cend), hi = min(lo + per, cend);
  int bad = 0;
  __syncthreads();
  for (int pb = lo; pb < hi; pb += kPiece) {
    const int pe = min(pb + kPiece, hi);
    warp_load(p.idx, pb, pe, pb, E, cache, bad);
    warp_count(pb, pe, pb, cache, wcnt + warp * E);
  }
  bad = __syncthreads_or(bad);
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = 0;
    for (int w = 0; w < W; ++w) {
      const int k = wcnt[w * E + e];
      wcnt[w * E + e] = run;
      run += k;
    }
    tot[e] = run;
  }
  if (threadIdx.x == 0) flag_s[0] = bad;
  cluster.sync();  // every CTA's totals are visible to the cluster
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
  int any_bad = 0;
  if (threadIdx.x < C) any_bad = *cluster.map_shared_rank(flag_s, static_cast<int>(threadIdx.x));
  any_bad = __syncthreads_or(any_bad);
  cluster.sync();  // no CTA reads another's shared memory after this point
  int P = 0, npad = 0;
  finalize_compute(p, cnt_s, off_s, pad_s, &P, &npad);
  finalize_write(p, cnt_s, off_s, pad_s, P, npad, any_bad, c, C);
  for (int i = threadIdx.x; i < W * E; i += blockDim.x) {
    const int e = i % E;
    wcnt[i] += off_s[e] + base[e];
  }
  __syncthreads();
  const bool cached = (hi - lo) <= kPiece;  // the one piece is still in the cache
  for (int pb = lo; pb < hi; pb += kPiece) {
    const int pe = min(pb + kPiece, hi);
    if (!cached) {
      int ignored = 0;
      warp_load(p.idx, pb, pe, pb, E, cache, ignored);
    }
    warp_assign(pb, pe, pb, cache, wcnt + warp * E, p.slot);
  }
}

// Shared set-up of the chunked kernels: load the chunk, count per warp.
struct ChunkCtx {
  int* wcnt;
  short* ecache;
  int cbase, lo, hi, bad;
};

__device__ __forceinline__ ChunkCtx chunk_count(const RouteParams& p, int* smem) {
  ChunkCtx c;
  const int W = blockDim.x >> 5, E = p.E, warp = threadIdx.x >> 5;
  c.wcnt = smem;
  c.ecache = reinterpret_cast<short*>(smem + W * E);
  c.cbase = blockIdx.x * p.chunk;
  const int cend = min(c.cbase + p.chunk, p.n);
  const int per = p.chunk / W;
  c.lo = min(c.cbase + warp * per, cend);
  c.hi = min(c.lo + per, cend);
  c.bad = 0;
  for (int i = threadIdx.x; i < W * E; i += blockDim.x) c.wcnt[i] = 0;
  warp_load(p.idx, c.lo, c.hi, c.cbase, E, c.ecache, c.bad);
  __syncthreads();
  warp_count(c.lo, c.hi, c.cbase, c.ecache, c.wcnt + warp * E);
  c.bad = __syncthreads_or(c.bad);
  return c;
}

__global__ void __launch_bounds__(512) ep_route_hist_kernel(RouteParams p) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ int smem[];
  const ChunkCtx c = chunk_count(p, smem);
  const int W = blockDim.x >> 5, E = p.E;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int s = 0;
    for (int w = 0; w < W; ++w) s += c.wcnt[w * E + e];
    p.hist[static_cast<size_t>(e) * p.nchunks + blockIdx.x] = s;
  }
  if (threadIdx.x == 0) p.badflag[blockIdx.x] = c.bad;
}

__global__ void __launch_bounds__(1024) ep_route_scan_kernel(RouteParams p) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ int smem[];
  const int E = p.E, NC = p.nchunks;
  int* cnt_s = smem;           // [E]
  int* off_s = cnt_s + E;      // [E+1]
  int* pad_s = off_s + E + 1;  // [E+1]
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  // Exclusive scan over chunks, one warp per expert: hist[e][c] becomes the
  // number of routes to e in chunks before c.
  for (int e = warp; e < E; e += nwarps) {
    int* row = p.hist + static_cast<size_t>(e) * NC;
    int carry = 0;
    for (int c0 = 0; c0 < NC; c0 += 128) {
      int v[4];
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int c = c0 + b * 32 + lane;
        v[b] = c < NC ? row[c] : 0;
      }
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        int x = v[b];
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
          const int y = __shfl_up_sync(kFull, x, d);
          if (lane >= d) x += y;
        }
        const int c = c0 + b * 32 + lane;
        if (c < NC) row[c] = carry + x - v[b];
        carry += __shfl_sync(kFull, x, 31);
      }
    }
    if (lane == 0) cnt_s[e] = carry;
  }
  int bad = 0;
  for (int c = threadIdx.x; c < NC; c += blockDim.x) bad |= p.badflag[c];
  bad = __syncthreads_or(bad);
  finalize(p, cnt_s, off_s, pad_s, bad);
}

__global__ void __launch_bounds__(512) ep_route_assign_kernel(RouteParams p) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ int smem[];
  const ChunkCtx c = chunk_count(p, smem);
  const int W = blockDim.x >> 5, E = p.E;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = p.offsets[e] + p.hist[static_cast<size_t>(e) * p.nchunks + blockIdx.x];
    for (int w = 0; w < W; ++w) {
      const int k = c.wcnt[w * E + e];
      c.wcnt[w * E + e] = run;
      run += k;
    }
  }
  __syncthreads();
  warp_assign(c.lo, c.hi, c.cbase, c.ecache, c.wcnt + (threadIdx.x >> 5) * E, p.slot);
}

}  // namespace

int cluster_warps(int E) {
  int w = 32;
  while (w > 1 && cluster_smem_bytes(w, E) > static_cast<size_t>(kSmemBudget) - 512) --w;
  return w;
}

int chunk_warps(int E) {
  return std::max(1, std::min(kChunkWarpsMax, 32768 / (4 * E)));
}

// Fails when this device cannot run the sm_103a image.
cudaError_t probe_kernel_image() {
  cudaFuncAttributes a;
  return cudaFuncGetAttributes(&a, ep_prepare_cluster_kernel);
}

cudaError_t launch_prepare(const RouteParams& p0, int num_sms, cudaStream_t s, int* launches) {
  RouteParams p = p0;
  *launches = 0;
  const int Wc = cluster_warps(p.E);
  if (p.n <= kMaxCluster * Wc * kClusterMaxPerWarp) {
    // Cluster size for about 64 routes per warp, then an even split in
    // multiples of 32 routes per warp.
    const long long per_cta = static_cast<long long>(Wc) * 64;
    int C = static_cast<int>(std::min<long long>(kMaxCluster, std::max<long long>(1, (p.n + per_cta - 1) / per_cta)));
    long long rpw = (p.n + static_cast<long long>(C) * Wc - 1) / (static_cast<long long>(C) * Wc);
    rpw = std::max<long long>(32, ((rpw + 31) / 32) * 32);
    p.warps = Wc;
    p.chunk = static_cast<int>(rpw * Wc);
    C = static_cast<int>(std::max<long long>(1, (p.n + p.chunk - 1) / p.chunk));
    p.nchunks = C;
    *launches = 1;
    return launch_pdl(ep_prepare_cluster_kernel, dim3(C), dim3(Wc * 32), cluster_smem_bytes(Wc, p.E),
                      s, static_cast<unsigned>(C), p);
  }
  // p.nchunks arrives as the capacity of hist (chunks); pick routes per warp
  // (a multiple of 32) for about two CTAs per SM without exceeding it.
  const int W = chunk_warps(p.E);
  const long long cap = p.nchunks;
  const long long target = std::min<long long>(cap, 2LL * num_sms);
  long long rpw = (p.n + target * W - 1) / (target * W);
  rpw = std::max<long long>(32, ((rpw + 31) / 32) * 32);
  while ((p.n + rpw * W - 1) / (rpw * W) > cap) rpw += 32;
  p.warps = W;
  p.chunk = static_cast<int>(rpw * W);
  p.nchunks = static_cast<int>((p.n + p.chunk - 1) / p.chunk);
  const size_t chunk_smem = static_cast<size_t>(W) * p.E * 4 + ((static_cast<size_t>(p.chunk) * 2 + 15) & ~static_cast<size_t>(15));
  const size_t scan_smem = static_cast<size_t>(3 * p.E + 2) * 4;
  if (chunk_smem > static_cast<size_t>(kSmemBudget) - 512) return cudaErrorInvalidConfiguration;
  cudaError_t e = launch_pdl(ep_route_hist_kernel, dim3(p.nchunks), dim3(W * 32), chunk_smem, s, 0u, p);
  if (e != cudaSuccess) return e;
  e = launch_pdl(ep_route_scan_kernel, dim3(1), dim3(1024), scan_smem, s, 0u, p);
  if (e != cudaSuccess) return e;
  e = launch_pdl(ep_route_assign_kernel, dim3(p.nchunks), dim3(W * 32), chunk_smem, s, 0u, p);
  *launches = 3;
  return e;
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

// Chunk plan for the fixed array: (E + 1) * chunks counters must fit in it,
// and a chunk's cached expert ids must fit in shared memory.  Returns false
// when no plan fits (the caller reports EP_ERR_LIMIT).
bool static_scratch_plan(int n, int E, int num_sms, int* warps, int* chunk, int* nchunks) {
  const int W = chunk_warps(E);
  const long long cap = kStaticScratchInts / (E + 1);
  if (cap < 1) return false;
  const long long target = std::min<long long>(cap, 2LL * num_sms);
  long long rpw = (n + target * W - 1) / (target * W);
  rpw = std::max<long long>(32, ((rpw + 31) / 32) * 32);
  while ((n + rpw * W - 1) / (rpw * W) > cap) rpw += 32;
  const long long ch = rpw * W;
  const size_t smem = static_cast<size_t>(W) * E * 4 + ((static_cast<size_t>(ch) * 2 + 15) & ~static_cast<size_t>(15));
  if (smem > static_cast<size_t>(kSmemBudget) - 512) return false;
  *warps = W;
  *chunk = static_cast<int>(ch);
  *nchunks = static_cast<int>(std::max(1LL, (n + ch - 1) / ch));
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
  const size_t chunk_smem = static_cast<size_t>(W) * p.E * 4 + ((static_cast<size_t>(p.chunk) * 2 + 15) & ~static_cast<size_t>(15));
  const size_t scan_smem = static_cast<size_t>(3 * p.E + 2) * 4;
  ep_route_hist_kernel<<<p.nchunks, W * 32, chunk_smem, s>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  ep_route_scan_kernel<<<1, 1024, scan_smem, s>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  ep_route_assign_kernel<<<p.nchunks, W * 32, chunk_smem, s>>>(p);
  *launches = 3;
  return cudaGetLastError();
}

}  // namespace ep
