// ep_internal.cuh -- declarations shared by libep's translation units.
//
// Handle memory layout (all int32 words, 256-byte aligned sections):
//   header   : [0] status bits, [1] T of the last prepare, [2] P (rows in use),
//              [3] number of padding rows, [4] alignment A, [5] valid routes V,
//              [6] kPreparedMagic once a prepare has written the header
//              (kTimedOutMagic after a grid-wide prepare gave up waiting),
//              [7] the chunked prepare's CTA ticket (zero between prepares),
//              [8] the grid-wide prepare's arrival word (its low 31 bits
//              zero between prepares)
//   counts   : c_e                     [E]
//   offsets  : off_e (padded, e=0..E)  [E+1]
//   slot     : receive row of route r  [max_tokens*K]
//   pad_list : padding rows, ascending [min(E*(max_alignment-1), R) or 1]
//   hist     : per-chunk expert counts, chunk-major [max_chunks][E]
//   badflag  : per-chunk "saw an index outside [-1,E)" [max_chunks]
//   dest     : sharded layers only, owner rank of route r [max_tokens*K]
// A sharded layer keeps its own experts' counts and offsets ([E/N], [E/N+1])
// and its own padding rows in the same sections.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "../../include/ep.h"

namespace ep {

enum HeaderWord { kHdrStatus = 0, kHdrT = 1, kHdrP = 2, kHdrNPad = 3, kHdrA = 4, kHdrV = 5,
                  kHdrMagic = 6, kHdrTicket = 7, kHdrBarrier = 8 };
constexpr int kPreparedMagic = 0x45505245;
constexpr int kTimedOutMagic = 0x45505454;  // a grid-wide prepare whose wait gave up
constexpr int kHeaderBytes = 256;

// Routing-map kernels keep their per-warp counters in shared memory and stay
// within the default 48 KB, so that no function attribute has to be set
// before a graph capture: dynamic shared memory up to kSmemBudget - 1 KB,
// the rest left to the kernels' small static arrays.
constexpr int kSmemBudget = 48 * 1024;
constexpr int kChunkWarpsMax = 16;
// prepare runs as one launch of a thread-block cluster (at most kMaxCluster
// CTAs exchanging per-expert totals through distributed shared memory) while
// it needs at most kMaxJ routes per lane, else as three kernels.  A lane keeps
// the expert ids of its routes in registers between counting and assigning.
constexpr int kMaxCluster = 8;          // portable cluster size
constexpr int kMaxClusterWide = 16;     // non-portable, where the device allows it
constexpr int kMaxJ = 16;  // routes per lane, 512 per warp
// The cluster's CTA count is chosen for kClusterRoutesPerWarp routes per
// warp; once all kMaxCluster CTAs are in use a warp takes up to 32 * kMaxJ.
// More CTAs mean fewer serial 32-route assignment steps per warp for a wider
// exchange of totals: a Mixtral-sized batch (8192 routes) took 9.5 us on 8
// CTAs (64 per warp), 10.5 on 4 and 11.0 on 2.
constexpr int kClusterRoutesPerWarp = 64;

// Programmatic dependent launch: every libep kernel is launched so that it may
// be scheduled while the previous kernel on the stream drains, and waits at
// its first instruction for that kernel to complete and its writes to be
// visible (griddepcontrol.wait), so no data is read or written early.  (The
// one thing done before the wait is an L2 prefetch of source rows by the
// dispatch scatter and the gather-sum, a hint that loads no row into the SM.)
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Launch with programmatic stream serialization; cluster > 0 adds a cluster
// dimension, cooperative = true asks for a cooperative launch (every block
// resident at once, so blocks may wait on one another).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_ex(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t s, unsigned cluster, bool cooperative, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[3];
  unsigned n = 0;
  at[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (cluster > 0) {
    at[n].id = cudaLaunchAttributeClusterDimension;
    at[n].val.clusterDim.x = cluster;
    at[n].val.clusterDim.y = 1;
    at[n].val.clusterDim.z = 1;
    ++n;
  }
  if (cooperative) {
    at[n].id = cudaLaunchAttributeCooperative;
    at[n].val.cooperative = 1;
    ++n;
  }
  cfg.attrs = at;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, unsigned cluster, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[2];
  unsigned n = 0;
  at[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (cluster > 0) {
    at[n].id = cudaLaunchAttributeClusterDimension;
    at[n].val.clusterDim.x = cluster;
    at[n].val.clusterDim.y = 1;
    at[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = at;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

struct Layout {
  size_t counts, offsets, slot, pad_list, hist, badflag, dest, total;
  size_t oidx, owner;  // rank-major layers: per-route owner ids (int64) and owners (int32)
  int64_t pad_cap;     // entries of pad_list
  int64_t max_chunks;  // chunk rows of hist
};

struct LayerInfo {
  ep_layer_config_t cfg;
  int64_t R;
  int es;  // payload element size in bytes
  Layout lay;
  int64_t nranks;  // sharded layers: N (0 for a single-buffer layer)
  int64_t rank;    // and this rank
  bool rank_major; // rank-major receive layout (ep_register_layer_rank_major)
};

// Routing-map parameters (one prepare call).
struct RouteParams {
  const long long* idx;  // [T*K]
  int n;                 // routes T*K
  int T, K, E, A;
  int a_log2;            // log2(A) when A is a power of two, else -1
  long long R;
  long long pad_cap;     // entries of pad_list
  int warps;             // warps per CTA
  int chunk;             // routes per CTA (multi-CTA path)
  int nchunks;           // CTAs of the multi-CTA path; hist row stride
  int* hdr;
  int* counts;           // handle copy of c_e
  int* counts_user;      // caller's token_counts
  int* offsets;          // [E+1]
  int* slot;             // [T*K]
  int* pad_list;
  int* hist;             // [E][nchunks]
  int* badflag;          // [nchunks]
  // Sharded layers (nranks > 0): all ranks' counts [nranks][E], this rank,
  // and the owner map [T*K] written next to the slot map.
  const int* all_counts;
  int nranks;
  int rank;
  int* dest;
  // Rank-major layers: the caller's topk_idx [T*K] (over E_all experts, eloc
  // per rank), turned into per-route owner ids oidx (the owner at the first
  // route of each owner in a token, -1 at the others, nranks for an invalid
  // index) and owners (every valid route's owner, -1 else).
  const long long* idx_in;
  long long* oidx;
  int* owner;
  int E_all, eloc;
};

// Row-kernel parameters (dispatch / combine / their backward passes).
struct RowParams {
  int* hdr;
  const int* slot;
  const int* pad_list;
  int T, K, H;
  int R;                 // receive rows; slots outside [0, R) are never followed
  int pad_cap;           // entries of pad_list
  int dtype;             // ep_dtype_t of the payload rows
  int rowbytes;          // H * element size (a multiple of 16)
  const void* src;
  void* dst;
  const float* w_in;
  float* w_out;
  const float* scale;    // weighted combine: recv_topk_weights [R]
  const void* aux;       // weighted combine backward: expert_out [R, H]
  int prefetch;          // scatter: L2-prefetch source rows before waiting
  int resident_warps;    // warps of the launch that fit on the GPU at once
  int tok_warps;         // scatter: warps [0, tok_warps) take one token item each;
                         // the others stride over the prepared padding items
  // Sharded layers: the owner map [T*K] and, per rank, the address of that
  // rank's receive-side buffer (dst_tab / src_tab: payload rows, wout_tab /
  // win_tab: per-row weights); this rank's own buffer is entry `rank`.
  const int* dest;
  int nranks;
  int rank;
  void* const* dst_tab;
  const void* const* src_tab;
  float* const* wout_tab;
  const float* const* win_tab;
  // Rank-major layers: topk_idx [T*K] and the all-route owner map; per owner
  // the address of its received rows' expert ids (idx_tab, int64 [rows][K]);
  // experts per rank.
  const long long* idx;
  const int* owner;
  long long* const* idx_tab;
  int eloc;
};

// Row kernels write nothing unless a prepare has written the header, and not
// after an overflowing prepare; they flag a token count that differs from the
// prepared one.  The header words are loaded first (load_header) and checked
// later (header_ok), so that a kernel can issue the loads of its first item
// in between: those loads stay inside the buffers whatever the header holds
// (slots are followed only inside [0, R), token rows are below T), and
// nothing is stored before the check.  rows_ok does both at once.
struct Header {
  int magic, status, npad, P, T;
};

__device__ __forceinline__ Header load_header(const RowParams& p) {
  Header h;
  h.magic = p.hdr[kHdrMagic];
  h.status = p.hdr[kHdrStatus];
  h.npad = p.hdr[kHdrNPad];
  h.P = p.hdr[kHdrP];
  h.T = p.hdr[kHdrT];
  return h;
}

// Returns true to proceed.
__device__ __forceinline__ bool header_ok(const Header& h, const RowParams& p) {
  if (h.magic != kPreparedMagic) return false;
  if (h.status & (EP_ST_OVERFLOW | EP_ST_COUNTS_MISMATCH)) return false;
  if (h.npad < 0 || h.npad > p.pad_cap || h.P > p.R) return false;
  if (h.T != p.T) {
    if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(&p.hdr[kHdrStatus], EP_ST_TOKENS_MISMATCH);
    return false;
  }
  return true;
}

__device__ __forceinline__ bool rows_ok(const RowParams& p) { return header_ok(load_header(p), p); }

// Resident blocks per SM of a kernel on the current device (cached).
int resident_blocks(const void* kern, int threads, size_t smem);

// Routing map: returns the first CUDA error, and the number of kernels launched.
// max_cluster: the largest cluster the one-launch prepare may use on the
// device (prepare_max_cluster()); wide_ctas: the most CTAs of the grid-wide
// prepare that fit on the device at once (prepare_wide_ctas()).
cudaError_t launch_prepare(const RouteParams& p, int num_sms, int max_cluster, int wide_ctas,
                           cudaStream_t s, int* launches);
// CTAs of the grid-wide prepare that fit on the current device at once
// (0 where it cannot run); host-side, called once per device.
int prepare_wide_ctas();
// Warps per CTA of the cluster / chunked routing kernels for E experts.
int cluster_warps(int E);
// True when prepare of n routes over E experts is the single cluster launch
// (a few CTAs, most SMs idle while it runs), false for the chunked kernels.
bool prepare_is_one_launch(long long n, int E, int max_cluster);
// Largest cluster of the prepare kernel the current device can run: 16 CTAs
// (a non-portable cluster size, allowed on the kernel here) when one such
// cluster fits on the device, else kMaxCluster.  Host-side; called once per
// device, before any per-step call.
int prepare_max_cluster();
int chunk_warps(int E);

// Sharded routing map: count = this rank's histogram only (written to
// p.counts_user); prepare = the slot and owner maps from the all-gathered
// counts p.all_counts.  One cluster launch of at most max_cluster CTAs.
cudaError_t launch_shard_count(const RouteParams& p, int max_cluster, cudaStream_t s, int* launches);
cudaError_t launch_shard_prepare(const RouteParams& p, int max_cluster, cudaStream_t s,
                                 int* launches);
// Largest batch (routes) the sharded routing map takes for E experts on a
// cluster of max_cluster CTAs.
long long shard_max_routes(int E, int max_cluster);
// Largest cluster of the sharded routing modes on the current device (16 or
// kMaxCluster); host-side, called once per device.
int shard_max_cluster();
// Rank-major layers: the per-route owner ids and owners of p.idx_in, written
// to p.oidx and p.owner (one launch, chained like the others).
cudaError_t launch_rank_major_owners(const RouteParams& p, int num_sms, cudaStream_t s);

// Fixed-array variant of the routing map (see ep_prepare_static_scratch):
// 2^18 ints = 1 MiB of per-chunk counters in a __device__ array.
constexpr int kStaticScratchInts = 1 << 18;
cudaError_t static_scratch_address(int** out);
bool static_scratch_plan(int n, int E, int num_sms, int* warps, int* chunk, int* nchunks);
cudaError_t launch_prepare_static_scratch(const RouteParams& p, int* scratch, int num_sms,
                                          cudaStream_t s, int* launches);

// dispatch (weights) and combine_bwd (no weights): token-major row scatter.
cudaError_t launch_scatter(const RowParams& p, bool weights, int npad_max, int num_sms,
                           cudaStream_t s);
// The same for a sharded layer: rows go to their owner's buffer through
// p.dst_tab (and weights through p.wout_tab); padding rows of this rank's own
// buffer are zeroed.
cudaError_t launch_scatter_sharded(const RowParams& p, bool weights, int npad_max, int num_sms,
                                   cudaStream_t s);
// combine / dispatch_bwd of a sharded layer: rows read from their owner's
// buffer through p.src_tab (weights through p.win_tab, which may be null).
cudaError_t launch_gather_sharded(const RowParams& p, bool weights, int num_sms, cudaStream_t s);
// Rank-major push (dispatch, combine_bwd): rows through p.dst_tab at the
// first route of each owner in a token; with p.idx_tab set (dispatch), each
// received row's K expert ids relative to its owner and weights (p.wout_tab,
// may be null) too.
cudaError_t launch_scatter_rank_major(const RowParams& p, int num_sms, cudaStream_t s);
// Rank-major dispatch_bwd: token gradients as the sharded gather-sum, weight
// gradients (p.w_out) from the owners' [rows][K] (p.win_tab, null for zeros).
cudaError_t launch_gather_rank_major_bwd(const RowParams& p, int num_sms, cudaStream_t s);

// combine (no weights) and dispatch_bwd (weights): per-token gather-sum;
// scaled: each row multiplied by its receive row's weight (weighted combine).
cudaError_t launch_gather(const RowParams& p, bool weights, bool scaled, int num_sms,
                          cudaStream_t s);
// Backward of the weighted combine: scaled token gradient to each slot, and
// the weight gradient <grad[t], expert_out[slot]> per receive row.
cudaError_t launch_combine_bwd_scaled(const RowParams& p, int npad_max, int num_sms,
                                      cudaStream_t s);

}  // namespace ep
