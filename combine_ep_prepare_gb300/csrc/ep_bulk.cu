// ep_bulk.cu -- row scatter of dispatch and combine_bwd with bulk copies
// (TMA, cp.async.bulk) on sm_103a.
//
// Same contract as the register scatter of ep_rows.cu (TransformerEngine PR
// #3034, "Per-step": nvte_ep_dispatch places each token row and its routing
// weight in its expert-major receive slots; nvte_ep_combine_bwd copies each
// token's gradient to its slots; padding rows become zeros), but the bytes
// never pass through registers: each warp streams its rows in 4 KB chunks from
// global to shared memory with one bulk load (completion counted by an
// mbarrier), then writes the chunk to each of the token's K receive rows with
// bulk shared-to-global stores.  One lane drives the copy engine; the load
// of the warp's next chunk is in flight while the current chunk's stores run.
// Padding chunks are stored from a zero-filled shared buffer.
//
// Waits: every mbarrier wait polls at most kWaitPolls times; if a load never
// completes, the kernel sets EP_ST_TIMEOUT in the handle's status word,
// waits once more (bounded) for its copies, and leaves.
#include "ep_internal.cuh"

namespace ep {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kChunk = 4096;       // bytes per item (a row is cut into chunks)
constexpr int kStages = 2;         // shared-memory chunks per warp
constexpr int kWarps = 4;          // warps per CTA
constexpr unsigned kWaitPolls = 1u << 20;     // a normal load completes in microseconds
constexpr unsigned kCleanupPolls = 1u << 14;

constexpr size_t bulk_smem_bytes() {
  return static_cast<size_t>(kChunk) * (1 + kWarps * kStages) + 8 * kWarps * kStages;
}

__device__ __forceinline__ unsigned smem_u32(const void* p) {
  return static_cast<unsigned>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, unsigned parity) {
  unsigned ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, unsigned parity,
                                                  unsigned polls = kWaitPolls) {
  for (unsigned i = 0; i < polls; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}
__device__ __forceinline__ void bulk_load(void* sdst, const void* gsrc, unsigned bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(sdst)),
      "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void bulk_store(void* gdst, const void* ssrc, unsigned bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst),
               "r"(smem_u32(ssrc)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// All but the most recent bulk-store group have finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read_but_last() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

template <bool WEIGHTS>
__global__ void __launch_bounds__(kWarps * 32) ep_scatter_bulk_kernel(RowParams p) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ __align__(128) unsigned char smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  unsigned char* zero = smem;
  unsigned char* stage = smem + kChunk * (1 + warp * kStages);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kChunk * (1 + kWarps * kStages)) + warp * kStages;
  for (int i = threadIdx.x; i < kChunk / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(zero)[i] = make_uint4(0u, 0u, 0u, 0u);
  if (lane == 0)
    for (int s = 0; s < kStages; ++s) mbar_init(&bars[s], 1);
  // The zeros (written by threads) and the barrier initialisation must be
  // visible to the copy engine before its first use.
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  __syncthreads();
  if (!rows_ok(p)) return;

  const int K = p.K;
  const long long rowbytes = static_cast<long long>(p.H) * 2;
  const unsigned cpr = static_cast<unsigned>((rowbytes + kChunk - 1) / kChunk);
  const unsigned rows = static_cast<unsigned>(p.T + p.hdr[kHdrNPad]);
  const unsigned items = rows * cpr;
  const unsigned gw = blockIdx.x * kWarps + warp, nw = gridDim.x * kWarps;
  const unsigned mine = items > gw ? (items - gw + nw - 1) / nw : 0u;
  const unsigned char* src = reinterpret_cast<const unsigned char*>(p.src);
  unsigned char* dst = reinterpret_cast<unsigned char*>(p.dst);

  // Lane 0's copy-engine state: parity of the next wait on each stage.
  // Loads run up to kStages - 1 chunks ahead of the stores.
  unsigned parity = 0;
  auto issue_load = [&](unsigned j) {  // lane 0 only
    const unsigned it = gw + j * nw;
    const unsigned row = it / cpr, ch = it - row * cpr;
    if (row >= static_cast<unsigned>(p.T)) return;  // padding: nothing to load
    const long long off = static_cast<long long>(ch) * kChunk;
    const unsigned bytes = static_cast<unsigned>(min(static_cast<long long>(kChunk), rowbytes - off));
    uint64_t* bar = &bars[j % kStages];
    mbar_expect_tx(bar, bytes);
    bulk_load(stage + (j % kStages) * kChunk, src + row * rowbytes + off, bytes, bar);
  };
  if (lane == 0)
    for (unsigned j = 0; j < kStages && j < mine; ++j) issue_load(j);

  bool failed = false;
  for (unsigned j = 0; j < mine; ++j) {
    const unsigned it = gw + j * nw;
    const unsigned row = it / cpr, ch = it - row * cpr;
    const long long off = static_cast<long long>(ch) * kChunk;
    const unsigned bytes = static_cast<unsigned>(min(static_cast<long long>(kChunk), rowbytes - off));
    const int s = static_cast<int>(j % kStages);
    if (row < static_cast<unsigned>(p.T)) {
      int my = lane < K ? __ldg(p.slot + static_cast<size_t>(row) * K + lane) : -1;
      if (static_cast<unsigned>(my) >= static_cast<unsigned>(p.R)) my = -1;
      if (WEIGHTS && ch == 0 && my >= 0) p.w_out[my] = __ldg(p.w_in + static_cast<size_t>(row) * K + lane);
      int ok = 1;
      if (lane == 0) {
        ok = mbar_wait_bounded(&bars[s], (parity >> s) & 1u) ? 1 : 0;
        if (ok) parity ^= 1u << s;
      }
      if (__shfl_sync(kFull, ok, 0) == 0) {
        failed = true;
        break;
      }
      for (int k = 0; k < K; ++k) {
        const int d = __shfl_sync(kFull, my, k);
        if (lane == 0 && d >= 0) bulk_store(dst + static_cast<long long>(d) * rowbytes + off, stage + s * kChunk, bytes);
      }
    } else {
      const int d = __ldg(p.pad_list + (row - p.T));
      if (static_cast<unsigned>(d) < static_cast<unsigned>(p.R)) {
        if (WEIGHTS && ch == 0 && lane == 0) p.w_out[d] = 0.0f;
        if (lane == 0) bulk_store(dst + static_cast<long long>(d) * rowbytes + off, zero, bytes);
      }
    }
    if (lane == 0) {
      bulk_commit();
      // The previous chunk's stage is refilled (with chunk j - 1 + kStages)
      // once the previous chunk's stores have read it; this chunk's stores
      // keep running meanwhile.
      if (j >= 1 && j - 1 + kStages < mine) {
        bulk_wait_read_but_last();
        issue_load(j - 1 + kStages);
      }
    }
    __syncwarp();
  }
  if (lane == 0) {
    if (failed) {
      atomicOr(&p.hdr[kHdrStatus], static_cast<int>(EP_ST_TIMEOUT));
      // Loads still in flight target this CTA's shared memory: give them one
      // more bounded wait before leaving.
      for (int s = 0; s < kStages; ++s) mbar_wait_bounded(&bars[s], (parity >> s) & 1u, kCleanupPolls);
    }
    bulk_wait_all();
  }
}

}  // namespace

cudaError_t launch_scatter_bulk(const RowParams& p, bool weights, int npad_max, int num_sms,
                                cudaStream_t s) {
  const long long rowbytes = static_cast<long long>(p.H) * 2;
  const long long cpr = (rowbytes + kChunk - 1) / kChunk;
  const long long items = (static_cast<long long>(p.T) + npad_max) * cpr;
  const void* kern = weights ? reinterpret_cast<const void*>(ep_scatter_bulk_kernel<true>)
                             : reinterpret_cast<const void*>(ep_scatter_bulk_kernel<false>);
  const int per_sm = resident_blocks(kern, kWarps * 32, bulk_smem_bytes());
  long long blocks = (items + kWarps - 1) / kWarps;
  const long long cap = static_cast<long long>(num_sms) * per_sm;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  if (weights)
    return launch_pdl(ep_scatter_bulk_kernel<true>, dim3(static_cast<unsigned>(blocks)), dim3(kWarps * 32),
                      bulk_smem_bytes(), s, 0u, p);
  return launch_pdl(ep_scatter_bulk_kernel<false>, dim3(static_cast<unsigned>(blocks)), dim3(kWarps * 32),
                    bulk_smem_bytes(), s, 0u, p);
}

}  // namespace ep
