// ep_rows.cu -- row-movement kernels of dispatch, combine and their backward
// passes (sm_103a).
//
// TransformerEngine PR #3034, "Expert Parallelism: common C API + NCCL EP
// backend", section "Per-step (allocation-free, CUDA-graph capturable)":
//   nvte_ep_dispatch     tokens and routing weights -> expert-major slots
//   nvte_ep_combine      unweighted sum of expert outputs back to the token
//   nvte_ep_dispatch_bwd token and weight gradients back to the token
//   nvte_ep_combine_bwd  token gradient to each slot; padded slots zeroed
// On one GPU every "send" is a row copy inside HBM, so two kernels cover all
// four calls:
//   scatter    (dispatch, combine_bwd): each source row is read ONCE and
//              written to its K receive rows; padding rows get zeros.
//   gather-sum (combine, dispatch_bwd): each token reads its K rows and sums
//              them in float32, k ascending from +0.0f, then rounds once to
//              the payload type (bf16 / fp16: round to nearest even; fp32:
//              the sum).  No atomics: the result does not depend on
//              scheduling.
//
// Both are HBM-bound (at most K adds per element).  Work is split into items
// of (row, column chunk); a warp moves one chunk with 16- or 32-byte vector
// accesses, each warp instruction touching 512 or 1024 contiguous bytes of
// one row.  The scatter's grid streams (one item per warp); the gather-sum's
// is persistent (the blocks that fit at once, striding over items) -- see
// launch_rows.  Rows are handled as bytes where no arithmetic is done
// (scatter) and as elements of the payload type where it is (gather-sum).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <map>
#include <mutex>
#include <utility>

#include "ep_internal.cuh"

namespace ep {
namespace {

constexpr unsigned kFull = 0xffffffffu;

// 16- or 32-byte vector of raw payload bits.  The 32-byte form uses the
// 256-bit global loads and stores of sm_100+ (half the instructions per byte).
template <int VB>
struct alignas(VB) Vec {
  unsigned w[VB / 4];
};

// Read-once streaming load (not kept in L1).
template <int VB>
__device__ __forceinline__ Vec<VB> ld_stream(const Vec<VB>* p);
template <>
__device__ __forceinline__ Vec<16> ld_stream<16>(const Vec<16>* p) {
  Vec<16> v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3])
               : "l"(p));
  return v;
}
template <>
__device__ __forceinline__ Vec<32> ld_stream<32>(const Vec<32>* p) {
  Vec<32> v;
  asm volatile("ld.global.nc.L1::no_allocate.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3]),
                 "=r"(v.w[4]), "=r"(v.w[5]), "=r"(v.w[6]), "=r"(v.w[7])
               : "l"(p));
  return v;
}

template <int VB>
__device__ __forceinline__ void st_vec(Vec<VB>* p, const Vec<VB>& v);
// 16 bytes: a plain store, which leaves the compiler free to schedule the
// surrounding loads (an asm store with a memory clobber measured 8% slower in
// the gather-sum).  32 bytes: the 256-bit store has no C++ spelling; the asm
// has no memory clobber for the same reason (no load in these kernels reads
// what a store of the same launch writes).
template <>
__device__ __forceinline__ void st_vec<16>(Vec<16>* p, const Vec<16>& v) {
  *reinterpret_cast<uint4*>(p) = make_uint4(v.w[0], v.w[1], v.w[2], v.w[3]);
}
template <>
__device__ __forceinline__ void st_vec<32>(Vec<32>* p, const Vec<32>& v) {
  asm volatile("st.global.v8.u32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(v.w[0]),
               "r"(v.w[1]), "r"(v.w[2]), "r"(v.w[3]), "r"(v.w[4]), "r"(v.w[5]), "r"(v.w[6]),
               "r"(v.w[7]));
}

template <int VB>
__device__ __forceinline__ Vec<VB> zero_vec() {
  Vec<VB> v;
#pragma unroll
  for (int i = 0; i < VB / 4; ++i) v.w[i] = 0u;
  return v;
}


// The K receive rows of a token, read by every lane of the warp (the same
// 4*K bytes: a broadcast), with 16- or 8-byte loads when K allows.  Entries
// k >= K, and rows outside [0, R), become -1.
template <int KMAX>
__device__ __forceinline__ void load_slots(const int* __restrict__ row, int K, int R, int (&s)[KMAX]) {
  if (K == KMAX && KMAX % 4 == 0) {
#pragma unroll
    for (int k = 0; k < KMAX; k += 4) {
      const int4 v = __ldg(reinterpret_cast<const int4*>(row) + k / 4);
      s[k] = v.x;
      s[k + 1] = v.y;
      s[k + 2] = v.z;
      s[k + 3] = v.w;
    }
  } else if (K == KMAX && KMAX % 2 == 0) {
#pragma unroll
    for (int k = 0; k < KMAX; k += 2) {
      const int2 v = __ldg(reinterpret_cast<const int2*>(row) + k / 2);
      s[k] = v.x;
      s[k + 1] = v.y;
    }
  } else {
#pragma unroll
    for (int k = 0; k < KMAX; ++k) s[k] = k < K ? __ldg(row + k) : -1;
  }
#pragma unroll
  for (int k = 0; k < KMAX; ++k)
    if (static_cast<unsigned>(s[k]) >= static_cast<unsigned>(R)) s[k] = -1;
}

// Entry i of a caller-owned device table of addresses (sharded layers).
template <typename Ptr>
__device__ __forceinline__ Ptr table_entry(const Ptr* tab, int i) {
  return reinterpret_cast<Ptr>(__ldg(reinterpret_cast<const unsigned long long*>(tab) + i));
}

// A row address taken from a table may be used only when it is 16-byte
// aligned (every vector access of the row kernels is); anything else is
// skipped and flagged in the status word instead of being dereferenced.
__device__ __forceinline__ bool usable_row_base(const void* b, int* hdr) {
  if (b != nullptr && (reinterpret_cast<uintptr_t>(b) & 15u) == 0) return true;
  atomicOr(hdr + kHdrStatus, static_cast<int>(EP_ST_BAD_POINTER));
  return false;
}

// Source rows of the scatter are the caller's token rows: which of them a
// warp copies does not depend on the routing map.  So, before it waits for
// the previous kernel, each warp asks L2 to fetch the chunks it will copy
// first, up to kPrefetchBytes / (K + 1) over the grid.  A bulk L2 prefetch is a hint: it moves no
// data into the SM and writes nothing, and the copies load the rows again
// after the wait, so it cannot change a result.  Addresses stay inside the
// T source rows; every chunk starts at a multiple of 16 bytes of a 16-byte
// aligned row and its size is a multiple of 16 bytes, as the bulk copy
// requires.
// The budget shrinks with K: after a warp has copied x bytes of prefetched
// rows it has also written K*x, so prefetched rows plus the writes that
// follow them stay within kPrefetchBytes, about three quarters of L2.
constexpr long long kPrefetchBytes = 96ll << 20;

__device__ __forceinline__ void prefetch_l2(const void* p, unsigned bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ void prefetch_first_chunks(const RowParams& p, int chunk_bytes, int cpr) {
  // Only the warps of the blocks that can be resident at once run while the
  // previous kernel does; they stride over the budget between them.
  const unsigned warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const unsigned nwarps = static_cast<unsigned>(p.resident_warps);
  if ((threadIdx.x & 31) != 0 || warp >= nwarps) return;
  const long long budget = kPrefetchBytes / (p.K + 1) / chunk_bytes;  // >= 1 (K <= 32)
  const unsigned items = static_cast<unsigned>(min(static_cast<long long>(p.T) * cpr, budget));
  const char* srcb = static_cast<const char*>(p.src);
  for (unsigned it = warp; it < items; it += nwarps) {
    const unsigned row = it / static_cast<unsigned>(cpr);
    const int off = static_cast<int>(it - row * static_cast<unsigned>(cpr)) * chunk_bytes;
    prefetch_l2(srcb + static_cast<size_t>(row) * p.rowbytes + off,
                static_cast<unsigned>(min(chunk_bytes, p.rowbytes - off)));
  }
}

// VB-byte vectors, U of them per lane per item (an item is 32*U*VB bytes of
// one row); K <= KMAX destinations per token.  Payload-type agnostic.
// PREFETCH instances serve dispatch behind the one-launch prepare, where most
// SMs idle while prepare runs.  combine_bwd normally follows combine, which
// keeps every SM busy, so it has no idle window to use.  The instances
// without the prefetch compile exactly as the plain scatter: with the
// prefetch code present but switched off by a flag, the compiler allocated
// registers differently and a Qwen3-sized step measured 4 us slower.
// SH (sharded layers): each route's row goes to its owner's buffer,
// p.dst_tab[owner] (its weight to p.wout_tab[owner]); padding rows belong to
// this rank's own buffer, entry p.rank.  No prefetch in these instances:
// their destinations may be another GPU's memory.
// RM (rank-major layers, with SH): the slot map holds a row only at the first
// route of each owner in a token; with the token's first chunk the warp also
// writes each such row's K expert ids relative to the owner (p.idx_tab) and
// weights (p.wout_tab, may be null): entry k is route k's where the owner
// holds its expert, -1 and 0.0f elsewhere.
template <int VB, int U, int KMAX, bool WEIGHTS, bool PREFETCH, bool SH = false, bool RM = false>
__global__ void __launch_bounds__(256) ep_scatter_rows_kernel(RowParams p) {
  using V = Vec<VB>;
  const int K = p.K, HV = p.rowbytes / VB;
  const int cpr = (HV + 32 * U - 1) / (32 * U);
  if (PREFETCH) prefetch_first_chunks(p, 32 * U * VB, cpr);
  pdl_wait();
  pdl_trigger();
  // The header is checked after a token item's slot and row loads are
  // issued (before any store); sharded instances and padding items check
  // it first.
  const Header hdr = load_header(p);
  if (SH && !header_ok(hdr, p)) return;
  const int lane = threadIdx.x & 31;
  const unsigned warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const unsigned nwarps = (gridDim.x * blockDim.x) >> 5;
  // Token items: one per warp of the first tok_warps.  Padding items (rows
  // T .. T + npad - 1 of the item space, npad as prepared): the remaining
  // warps, one item each as launched (the stride covers the worst case).
  const unsigned tok_items = static_cast<unsigned>(p.T) * static_cast<unsigned>(cpr);
  const unsigned tok_warps = static_cast<unsigned>(p.tok_warps);
  unsigned first, end, stride;
  if (warp < tok_warps) {
    first = warp;
    end = min(warp + 1u, tok_items);
    stride = 1u;
  } else {
    if (!SH && !header_ok(hdr, p)) return;
    const unsigned npad = static_cast<unsigned>(hdr.npad);
    first = tok_items + (warp - tok_warps);
    end = tok_items + npad * static_cast<unsigned>(cpr);
    stride = nwarps - tok_warps;
  }
  const char* srcb = static_cast<const char*>(p.src);
  char* dstb = static_cast<char*>(p.dst);
  for (unsigned it = first; it < end; it += stride) {
    const int row = static_cast<int>(it / cpr);
    const int ch = static_cast<int>(it - static_cast<unsigned>(row) * cpr);
    const int v0 = ch * 32 * U + lane;
    if (row < p.T) {
      int sl[KMAX];
      load_slots<KMAX>(p.slot + static_cast<size_t>(row) * K, K, p.R, sl);
      int ow[KMAX];
      if (SH) load_slots<KMAX>(p.dest + static_cast<size_t>(row) * K, K, p.nranks, ow);
      const V* src = reinterpret_cast<const V*>(srcb + static_cast<size_t>(row) * p.rowbytes);
      V buf[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int v = v0 + u * 32;
        if (v < HV) buf[u] = ld_stream<VB>(src + v);
      }
      if (!SH && !header_ok(hdr, p)) return;  // a token warp takes one item
      if (RM && ch == 0 && p.idx_tab != nullptr) {
        long long e = -1;
        float w = 0.0f;
        if (lane < K) {
          e = __ldg(p.idx + static_cast<size_t>(row) * K + lane);
          if (p.w_in != nullptr) w = __ldg(p.w_in + static_cast<size_t>(row) * K + lane);
        }
        const long long E_all = static_cast<long long>(p.eloc) * p.nranks;
        const int mine = (e >= 0 && e < E_all) ? static_cast<int>(e / p.eloc) : -1;
#pragma unroll
        for (int j = 0; j < KMAX; ++j) {
          if (sl[j] < 0 || ow[j] < 0 || lane >= K) continue;  // every lane holds all K slots
          const size_t at = static_cast<size_t>(sl[j]) * K + lane;
          long long* ib = table_entry(p.idx_tab, ow[j]);
          if (usable_row_base(ib, p.hdr)) ib[at] = mine == ow[j] ? e - static_cast<long long>(ow[j]) * p.eloc : -1LL;
          if (p.wout_tab != nullptr) {
            float* wb = table_entry(p.wout_tab, ow[j]);
            if (usable_row_base(wb, p.hdr)) wb[at] = mine == ow[j] ? w : 0.0f;
          }
        }
      }
      if (WEIGHTS && ch == 0 && lane < K) {
        const int my = __ldg(p.slot + static_cast<size_t>(row) * K + lane);
        if (static_cast<unsigned>(my) < static_cast<unsigned>(p.R)) {
          if (SH) {
            const int mo = __ldg(p.dest + static_cast<size_t>(row) * K + lane);
            if (static_cast<unsigned>(mo) < static_cast<unsigned>(p.nranks)) {
              float* wb = table_entry(p.wout_tab, mo);
              if (usable_row_base(wb, p.hdr)) wb[my] = __ldg(p.w_in + static_cast<size_t>(row) * K + lane);
            }
          } else {
            p.w_out[my] = __ldg(p.w_in + static_cast<size_t>(row) * K + lane);
          }
        }
      }
#pragma unroll
      for (int k = 0; k < KMAX; ++k) {
        if (sl[k] < 0) continue;  // masked route, or k >= K
        char* rb = dstb;
        if (SH) {
          if (ow[k] < 0) continue;
          rb = static_cast<char*>(table_entry(p.dst_tab, ow[k]));
          if (!usable_row_base(rb, p.hdr)) continue;
        }
        V* dst = reinterpret_cast<V*>(rb + static_cast<size_t>(sl[k]) * p.rowbytes);
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int v = v0 + u * 32;
          if (v < HV) st_vec<VB>(dst + v, buf[u]);
        }
      }
    } else {
      const int d = __ldg(p.pad_list + (row - p.T));
      if (static_cast<unsigned>(d) >= static_cast<unsigned>(p.R)) continue;
      char* rb = dstb;
      if (SH) {
        rb = static_cast<char*>(table_entry(p.dst_tab, p.rank));
        if (!usable_row_base(rb, p.hdr)) continue;
      }
      if (WEIGHTS && ch == 0 && lane == 0) {
        if (SH) {
          float* wb = table_entry(p.wout_tab, p.rank);
          if (usable_row_base(wb, p.hdr)) wb[d] = 0.0f;
        } else {
          p.w_out[d] = 0.0f;
        }
      }
      V* dst = reinterpret_cast<V*>(rb + static_cast<size_t>(d) * p.rowbytes);
      const V z = zero_vec<VB>();
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int v = v0 + u * 32;
        if (v < HV) st_vec<VB>(dst + v, z);
      }
    }
  }
}

// Payload element types of a 16-byte vector: unpack to float32 (exact) and
// pack from float32 (round to nearest even for bf16 / fp16).
template <int DT>
struct Elems;
template <>
struct Elems<EP_DTYPE_BF16> {
  static constexpr int kN = 8;
  __device__ static __forceinline__ void unpack(const Vec<16>& v, float (&f)[kN]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(v.w[i] << 16);
      f[2 * i + 1] = __uint_as_float(v.w[i] & 0xffff0000u);
    }
  }
  __device__ static __forceinline__ Vec<16> pack(const float (&f)[kN]) {
    Vec<16> o;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);  // .x low half
      o.w[i] = *reinterpret_cast<const unsigned*>(&h);
    }
    return o;
  }
};
template <>
struct Elems<EP_DTYPE_FP16> {
  static constexpr int kN = 8;
  __device__ static __forceinline__ void unpack(const Vec<16>& v, float (&f)[kN]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __half2float(__ushort_as_half(static_cast<unsigned short>(v.w[i] & 0xffffu)));
      f[2 * i + 1] = __half2float(__ushort_as_half(static_cast<unsigned short>(v.w[i] >> 16)));
    }
  }
  __device__ static __forceinline__ Vec<16> pack(const float (&f)[kN]) {
    Vec<16> o;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __half2 h = __floats2half2_rn(f[2 * i], f[2 * i + 1]);  // .x low half
      o.w[i] = *reinterpret_cast<const unsigned*>(&h);
    }
    return o;
  }
};
template <>
struct Elems<EP_DTYPE_FP32> {
  static constexpr int kN = 4;
  __device__ static __forceinline__ void unpack(const Vec<16>& v, float (&f)[kN]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) f[i] = __uint_as_float(v.w[i]);
  }
  __device__ static __forceinline__ Vec<16> pack(const float (&f)[kN]) {
    Vec<16> o;
#pragma unroll
    for (int i = 0; i < 4; ++i) o.w[i] = __float_as_uint(f[i]);
    return o;
  }
};

// KMAX >= K routes per token are loaded before any add, so that all of a
// token's row reads are in flight together.  SCALE: each row is first
// multiplied by its receive row's weight p.scale[slot] (a float32 product,
// then the float32 sum), the weighted combine.
// Before it waits for the previous kernel (whose tail leaves SMs idle), each
// warp asks L2 for the K row chunks of its first item.  The slot map comes
// from prepare, which ran before the previous kernel; should it still be in
// flight, a slot read here is merely stale, and a slot is followed only
// inside [0, R), so the worst case is a useless prefetch of a row of the
// caller's buffer.  A hint: nothing is loaded into the SM or written before
// the wait.  Measured in the step: Mixtral-like combine + dispatch_bwd 3.4 us
// shorter, decode 1.8 us; no change at DeepSeek-V3 size.
template <int U>
__device__ __forceinline__ void gather_prefetch_first(const RowParams& p) {
  const int lane = threadIdx.x & 31;
  const unsigned warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int HV = p.rowbytes >> 4;
  const int cpr = (HV + 32 * U - 1) / (32 * U);
  const unsigned t = warp / static_cast<unsigned>(cpr);
  if (t >= static_cast<unsigned>(p.T) || lane >= p.K) return;
  const int ch = static_cast<int>(warp - t * static_cast<unsigned>(cpr));
  const int my = __ldg(p.slot + static_cast<size_t>(t) * p.K + lane);
  if (static_cast<unsigned>(my) >= static_cast<unsigned>(p.R)) return;
  const int off = ch * 32 * U * 16;
  prefetch_l2(static_cast<const char*>(p.src) + static_cast<size_t>(my) * p.rowbytes + off,
              static_cast<unsigned>(min(32 * U * 16, p.rowbytes - off)));
}

// SH (sharded layers): route k's row is read from its owner's buffer,
// p.src_tab[owner] (the weight gradient from p.win_tab[owner]); lane k forms
// the row's address and hands it to the warp.  No prefetch in these
// instances: their sources may be another GPU's memory.
// RM (rank-major layers, with SH and WEIGHTS): the weight gradient of route k
// is entry k of its owner's row of the token, the row held at the owner's
// first route in the token (the lowest lane with the same owner, p.owner).
template <int DT, int KMAX, int U, bool WEIGHTS, bool SCALE, bool SH = false, bool RM = false>
__global__ void __launch_bounds__(256) ep_gather_sum_kernel(RowParams p) {
  if (!SH) gather_prefetch_first<U>(p);
  pdl_wait();
  pdl_trigger();
  // The header is checked once the first item's slot and row loads are
  // issued, before any store (sharded instances: first).
  const Header hdr = load_header(p);
  if (SH && !header_ok(hdr, p)) return;
  bool checked = SH;
  using El = Elems<DT>;
  constexpr int N = El::kN;
  const int lane = threadIdx.x & 31;
  const unsigned warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const unsigned nwarps = (gridDim.x * blockDim.x) >> 5;
  const int K = p.K, HV = p.rowbytes >> 4;
  const int cpr = (HV + 32 * U - 1) / (32 * U);
  const unsigned items = static_cast<unsigned>(p.T) * static_cast<unsigned>(cpr);
  const char* srcb = static_cast<const char*>(p.src);
  char* dstb = static_cast<char*>(p.dst);
  // (Loading a warp's next slots one iteration ahead measured slower:
  // DeepSeek-V3-like combine 313.9 -> 320.1 us, 6 more registers.)
  for (unsigned it = warp; it < items; it += nwarps) {
    const int t = static_cast<int>(it / cpr);
    const int ch = static_cast<int>(it - static_cast<unsigned>(t) * cpr);
    const int v0 = ch * 32 * U + lane;
    int my = lane < K ? __ldg(p.slot + static_cast<size_t>(t) * K + lane) : -1;
    if (static_cast<unsigned>(my) >= static_cast<unsigned>(p.R)) my = -1;
    const int my_slot = my;  // RM: this lane's row before the table checks below
    const char* mybase = srcb;  // SH: base of this lane's route's owner buffer
    int mo = 0;
    if (SH) {
      mo = lane < K ? __ldg(p.dest + static_cast<size_t>(t) * K + lane) : -1;
      if (static_cast<unsigned>(mo) >= static_cast<unsigned>(p.nranks)) my = -1;
      mybase = nullptr;
      if (my >= 0) {
        mybase = static_cast<const char*>(table_entry(p.src_tab, mo));
        if (!usable_row_base(mybase, p.hdr)) my = -1;
      }
    }
    float wgrad = 0.0f;  // weight gradient of this lane's route (WEIGHTS), stored below
    if (RM && WEIGHTS && ch == 0) {
      const int q = lane < K ? __ldg(p.owner + static_cast<size_t>(t) * K + lane) : -1;
      const unsigned same = __match_any_sync(kFull, q);
      const int rrow = __shfl_sync(kFull, my_slot, __ffs(same) - 1);
      if (lane < K && p.win_tab != nullptr && static_cast<unsigned>(q) < static_cast<unsigned>(p.nranks) &&
          rrow >= 0) {
        const float* wb = table_entry(p.win_tab, q);
        if (usable_row_base(wb, p.hdr)) wgrad = __ldg(wb + static_cast<size_t>(rrow) * K + lane);
      }
    } else if (WEIGHTS && ch == 0 && lane < K) {
      if (SH) {
        if (my >= 0 && p.win_tab != nullptr) {
          const float* wb = table_entry(p.win_tab, mo);
          if (usable_row_base(wb, p.hdr)) wgrad = __ldg(wb + my);
        }
      } else if (my >= 0 && p.w_in != nullptr) {
        wgrad = __ldg(p.w_in + my);
      }
    }
    float wk = 0.0f;
    if (SCALE && my >= 0) wk = __ldg(p.scale + my);
    // Lane k holds slot k; a shuffle hands each slot to the whole warp (this
    // measured faster here than every lane loading the K slots itself).
    int s[KMAX];
    float sc[KMAX];
    Vec<16> buf[KMAX][U];
#pragma unroll
    for (int k = 0; k < KMAX; ++k) {
      s[k] = __shfl_sync(kFull, my, k);  // lanes >= K hold -1
      sc[k] = SCALE ? __shfl_sync(kFull, wk, k) : 1.0f;
      const char* kb = srcb;
      if (SH) {
        const unsigned long long a = reinterpret_cast<unsigned long long>(mybase);
        const unsigned lo32 = __shfl_sync(kFull, static_cast<unsigned>(a), k);
        const unsigned hi32 = __shfl_sync(kFull, static_cast<unsigned>(a >> 32), k);
        kb = reinterpret_cast<const char*>((static_cast<unsigned long long>(hi32) << 32) | lo32);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) buf[k][u] = zero_vec<16>();
      if (s[k] >= 0) {
        const Vec<16>* src = reinterpret_cast<const Vec<16>*>(kb + static_cast<size_t>(s[k]) * p.rowbytes);
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int v = v0 + u * 32;
          if (v < HV) buf[k][u] = ld_stream<16>(src + v);
        }
      }
    }
    if (!checked) {
      if (!header_ok(hdr, p)) return;
      checked = true;
    }
    if (WEIGHTS && ch == 0 && lane < K) p.w_out[static_cast<size_t>(t) * K + lane] = wgrad;
    float acc[U][N];
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int j = 0; j < N; ++j) acc[u][j] = 0.0f;
#pragma unroll
    for (int k = 0; k < KMAX; ++k) {
      if (s[k] < 0) continue;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        float f[N];
        El::unpack(buf[k][u], f);
#pragma unroll
        for (int j = 0; j < N; ++j)
          acc[u][j] = __fadd_rn(acc[u][j], SCALE ? __fmul_rn(sc[k], f[j]) : f[j]);
      }
    }
    Vec<16>* dst = reinterpret_cast<Vec<16>*>(dstb + static_cast<size_t>(t) * p.rowbytes);
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int v = v0 + u * 32;
      if (v < HV) st_vec<16>(dst + v, El::pack(acc[u]));
    }
  }
}

// Backward of the weighted combine (result[t] = sum_k w[slot] * expert_out[slot]):
//   grad_expert_out[slot] = round( float32(w[slot] * grad[t]) )
//   g_w[slot]             = sum over h of grad[t][h] * expert_out[slot][h]
// One CTA per row (grid-stride): its threads split the row into 16-byte
// vectors, each thread keeps K partial dot products (float32 fused
// multiply-adds; for 16-bit payloads every product is exact), a warp reduces
// them by a fixed butterfly, and thread k adds the warps' sums in warp order
// -- the result does not depend on scheduling.  Padding rows get zeros.
// MINB = resident blocks per SM the registers are sized for (2 blocks of 256
// threads = 128 registers each).  K=8 has two instances: at 2 blocks per SM
// (126 registers) and at 3 (80 registers).  With a row of at most one
// 16-byte vector per thread (H <= 2048 in 16-bit types) the 3-block instance
// measured 13% faster (Qwen3-like layer: 101.7 against 116.6 us); with longer
// rows, which each thread walks in several steps, it measured 6% slower
// (DeepSeek-V3-like: 704 against 666 us), so those keep the 2-block one.
template <int DT, int KMAX, int MINB>
__global__ void __launch_bounds__(256, MINB) ep_combine_bwd_scaled_kernel(RowParams p) {
  pdl_wait();
  pdl_trigger();
  if (!rows_ok(p)) return;
  using El = Elems<DT>;
  constexpr int N = El::kN;
  __shared__ float part[2][8][KMAX];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const int K = p.K, HV = p.rowbytes >> 4;
  const unsigned rows = static_cast<unsigned>(p.T + p.hdr[kHdrNPad]);
  const char* srcb = static_cast<const char*>(p.src);
  const char* auxb = static_cast<const char*>(p.aux);
  char* dstb = static_cast<char*>(p.dst);
  int pb = 0;  // partial-sum buffer; alternates between consecutive token rows
  for (unsigned row = blockIdx.x; row < rows; row += gridDim.x) {
    if (row < static_cast<unsigned>(p.T)) {
      int my = lane < K ? __ldg(p.slot + static_cast<size_t>(row) * K + lane) : -1;
      if (static_cast<unsigned>(my) >= static_cast<unsigned>(p.R)) my = -1;
      const float wk = my >= 0 ? __ldg(p.scale + my) : 0.0f;
      int s[KMAX];
      float sc[KMAX], dp[KMAX];
#pragma unroll
      for (int k = 0; k < KMAX; ++k) {
        s[k] = __shfl_sync(kFull, my, k);
        sc[k] = __shfl_sync(kFull, wk, k);
        dp[k] = 0.0f;
      }
      const Vec<16>* g = reinterpret_cast<const Vec<16>*>(srcb + static_cast<size_t>(row) * p.rowbytes);
      for (int v = threadIdx.x; v < HV; v += blockDim.x) {
        float gf[N];
        El::unpack(ld_stream<16>(g + v), gf);
        Vec<16> xv[KMAX];
#pragma unroll
        for (int k = 0; k < KMAX; ++k) {
          xv[k] = zero_vec<16>();
          if (s[k] >= 0)
            xv[k] = ld_stream<16>(reinterpret_cast<const Vec<16>*>(auxb + static_cast<size_t>(s[k]) * p.rowbytes) + v);
        }
#pragma unroll
        for (int k = 0; k < KMAX; ++k) {
          if (s[k] < 0) continue;
          float xf[N], of[N];
          El::unpack(xv[k], xf);
#pragma unroll
          for (int j = 0; j < N; ++j) {
            of[j] = __fmul_rn(sc[k], gf[j]);
            dp[k] = __fmaf_rn(gf[j], xf[j], dp[k]);
          }
          st_vec<16>(reinterpret_cast<Vec<16>*>(dstb + static_cast<size_t>(s[k]) * p.rowbytes) + v,
                     El::pack(of));
        }
      }
#pragma unroll
      for (int k = 0; k < KMAX; ++k) {
        float x = dp[k];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(kFull, x, off);
        if (lane == 0) part[pb][warp][k] = x;
      }
      __syncthreads();
      if (static_cast<int>(threadIdx.x) < K && my >= 0) {
        float tot = 0.0f;
        for (int w = 0; w < nw; ++w) tot += part[pb][w][threadIdx.x];
        p.w_out[my] = tot;
      }
      pb ^= 1;
    } else {
      const int d = __ldg(p.pad_list + (row - p.T));
      if (static_cast<unsigned>(d) >= static_cast<unsigned>(p.R)) continue;
      Vec<16>* dst = reinterpret_cast<Vec<16>*>(dstb + static_cast<size_t>(d) * p.rowbytes);
      for (int v = threadIdx.x; v < HV; v += blockDim.x) st_vec<16>(dst + v, zero_vec<16>());
      if (threadIdx.x == 0) p.w_out[d] = 0.0f;
    }
  }
}

}  // namespace

// Resident blocks per SM of a row kernel on the current device, cached per
// (device, kernel): the occupancy query is host-side arithmetic, but it is
// kept off the per-step path.
int resident_blocks(const void* kern, int threads, size_t smem) {
  static std::mutex mu;
  static std::map<std::pair<int, const void*>, int> cache;
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find({dev, kern});
  if (it != cache.end()) return it->second;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, threads, smem) != cudaSuccess) {
    cudaGetLastError();
    n = 1;
  }
  n = std::max(1, n);
  cache[{dev, kern}] = n;
  return n;
}

namespace {

// Grid of a row kernel, one warp per item.  Persistent: at most the blocks
// that fit on the GPU at once, each warp striding over items (the gather-sum
// and the weighted backward).  Streaming: one item per warp, the hardware
// scheduler starting blocks as others finish (the scatter).  For the scatter
// the streaming grid measured 9-13% faster (DeepSeek-V3-like dispatch 397 ->
// 360 us, Qwen3-like 61 -> 54 us): every SM works on a narrow window of rows
// that advances through the batch, where persistent warps drift apart and
// widen the window of rows being written.  The gather-sum measured 2-5%
// slower streaming, so it stays persistent.
template <typename Kern>
cudaError_t launch_rows(Kern kern, RowParams p, long long items, int num_sms, cudaStream_t s,
                        bool persistent) {
  constexpr int kThreads = 256;
  const int per_sm = resident_blocks(reinterpret_cast<const void*>(kern), kThreads, 0);
  const long long want = std::max(1LL, (items + (kThreads / 32) - 1) / (kThreads / 32));
  const long long cap = static_cast<long long>(num_sms) * per_sm;
  // A persistent grid with fewer than 16 items per warp ends in a tail where
  // a few warps still work while others have none; twice the resident blocks
  // (the second set starts as the first finishes) shortened the Mixtral-sized
  // step by 2.3 us (combine and dispatch_bwd) and changed nothing at larger
  // sizes, where the cap stays at what fits.
  const long long capx = (persistent && want < 16 * cap) ? 2 * cap : cap;
  const long long blocks = persistent ? std::min(want, capx) : want;  // < 2^28 (registration)
  p.resident_warps = static_cast<int>(std::min(blocks, cap) * (kThreads / 32));
  return launch_pdl(kern, dim3(static_cast<unsigned>(blocks)), dim3(kThreads), 0, s, 0u, p);
}

// Grid of the scatter: one block per 8 token items, then one block per 8
// padding items of the worst-case padding, every warp taking at most one
// item (streaming); warps past the prepared padding exit at once.  The host
// cannot know the prepared padding without a synchronisation.  Capping the
// padding blocks at two per SM (the warps then striding over the prepared
// padding) measured slower, A/B in one process on one GB300: DeepSeek-V3-like
// step 1336 -> 1351 us, Qwen3-like 208 -> 213 us, while the ~8K exit-only
// blocks of the worst-case grid cost nothing measurable.
template <typename Kern>
cudaError_t launch_scatter_grid(Kern kern, RowParams p, long long cpr, int npad_max, int num_sms,
                                cudaStream_t s) {
  constexpr int kThreads = 256, kWarps = kThreads / 32;
  const int per_sm = resident_blocks(reinterpret_cast<const void*>(kern), kThreads, 0);
  const long long tok_blocks = (static_cast<long long>(p.T) * cpr + kWarps - 1) / kWarps;
  const long long pad_need = (static_cast<long long>(npad_max) * cpr + kWarps - 1) / kWarps;
  const long long pad_blocks = pad_need;
  const long long blocks = std::max(1LL, tok_blocks + pad_blocks);  // < 2^28 (registration)
  p.tok_warps = static_cast<int>(tok_blocks * kWarps);
  p.resident_warps = static_cast<int>(std::min<long long>(blocks, static_cast<long long>(num_sms) * per_sm) * kWarps);
  return launch_pdl(kern, dim3(static_cast<unsigned>(blocks)), dim3(kThreads), 0, s, 0u, p);
}

template <int VB, int U, int KMAX>
cudaError_t scatter_v(const RowParams& p, bool weights, int npad_max, int num_sms, cudaStream_t s) {
  const long long HV = p.rowbytes / VB;
  const long long cpr = (HV + 32 * U - 1) / (32 * U);
  if (weights && p.prefetch)
    return launch_scatter_grid(ep_scatter_rows_kernel<VB, U, KMAX, true, true>, p, cpr, npad_max, num_sms, s);
  if (weights)
    return launch_scatter_grid(ep_scatter_rows_kernel<VB, U, KMAX, true, false>, p, cpr, npad_max, num_sms, s);
  return launch_scatter_grid(ep_scatter_rows_kernel<VB, U, KMAX, false, false>, p, cpr, npad_max, num_sms, s);
}

template <int VB, int U>
cudaError_t scatter_k(const RowParams& p, bool weights, int npad_max, int num_sms, cudaStream_t s) {
  if (p.K <= 2) return scatter_v<VB, U, 2>(p, weights, npad_max, num_sms, s);
  if (p.K <= 4) return scatter_v<VB, U, 4>(p, weights, npad_max, num_sms, s);
  if (p.K <= 8) return scatter_v<VB, U, 8>(p, weights, npad_max, num_sms, s);
  if (p.K <= 16) return scatter_v<VB, U, 16>(p, weights, npad_max, num_sms, s);
  return scatter_v<VB, U, 32>(p, weights, npad_max, num_sms, s);
}

template <int DT, int KMAX, int U>
cudaError_t gather_k(const RowParams& p, bool weights, bool scaled, int num_sms, cudaStream_t s) {
  const int HV = p.rowbytes >> 4;
  const long long cpr = (HV + 32 * U - 1) / (32 * U);
  const long long items = static_cast<long long>(p.T) * cpr;
  if (scaled) return launch_rows(ep_gather_sum_kernel<DT, KMAX, U, false, true>, p, items, num_sms, s, true);
  if (weights) return launch_rows(ep_gather_sum_kernel<DT, KMAX, U, true, false>, p, items, num_sms, s, true);
  return launch_rows(ep_gather_sum_kernel<DT, KMAX, U, false, false>, p, items, num_sms, s, true);
}

template <int DT>
cudaError_t gather_dt(const RowParams& p, bool weights, bool scaled, int num_sms, cudaStream_t s) {
  if (p.K <= 2) return gather_k<DT, 2, 2>(p, weights, scaled, num_sms, s);  // U=4: 1 us slower (Mixtral step)
  if (p.K <= 4) return gather_k<DT, 4, 4>(p, weights, scaled, num_sms, s);
  if (p.K <= 8) return gather_k<DT, 8, 2>(p, weights, scaled, num_sms, s);
  if (p.K <= 16) return gather_k<DT, 16, 1>(p, weights, scaled, num_sms, s);
  return gather_k<DT, 32, 1>(p, weights, scaled, num_sms, s);
}

template <int DT>
cudaError_t combine_bwd_scaled_dt(const RowParams& p, int npad_max, int num_sms, cudaStream_t s) {
  // One CTA per row: items counted in warps for launch_rows.
  const long long rows8 = (static_cast<long long>(p.T) + npad_max) * 8;
  if (p.K <= 2) return launch_rows(ep_combine_bwd_scaled_kernel<DT, 2, 5>, p, rows8, num_sms, s, true);
  if (p.K <= 4) return launch_rows(ep_combine_bwd_scaled_kernel<DT, 4, 3>, p, rows8, num_sms, s, true);
  if (p.K <= 8) {
    if (p.rowbytes / 16 <= 256) return launch_rows(ep_combine_bwd_scaled_kernel<DT, 8, 3>, p, rows8, num_sms, s, true);
    return launch_rows(ep_combine_bwd_scaled_kernel<DT, 8, 2>, p, rows8, num_sms, s, true);
  }
  if (p.K <= 16) return launch_rows(ep_combine_bwd_scaled_kernel<DT, 16, 2>, p, rows8, num_sms, s, true);
  return launch_rows(ep_combine_bwd_scaled_kernel<DT, 32, 1>, p, rows8, num_sms, s, true);
}

}  // namespace

cudaError_t launch_scatter(const RowParams& p, bool weights, int npad_max, int num_sms,
                           cudaStream_t s) {
  // 32-byte vectors when every row starts on a 32-byte boundary.
  const bool v32 = (p.rowbytes % 32 == 0) && (reinterpret_cast<uintptr_t>(p.src) % 32 == 0) &&
                   (reinterpret_cast<uintptr_t>(p.dst) % 32 == 0);
  // Rows longer than 8 KB move 4 KB per warp item (DeepSeek-V3-like step 1.349 -> 1.331 ms);
  // shorter rows keep 2 KB items (no gain at 4 KB rows, 0.7 us slower at 8 KB).
  // A batch too small to give every SM two blocks of 4 KB / 2 KB items (a
  // decode step: 128 tokens of 14 KB rows made 64 blocks) moves 512-byte
  // items instead: decode-sized step 25.4 -> 22.7 us (dispatch 5.6 -> 4.2 us,
  // combine_bwd 4.5 -> 3.9 us; A/B in one process).
  const long long big_item = (v32 && p.rowbytes > 8192) ? 4096 : 2048;
  const long long small_items = static_cast<long long>(p.T) * ((p.rowbytes + 511) / 512);
  const long long big_items = static_cast<long long>(p.T) * ((p.rowbytes + big_item - 1) / big_item);
  if (big_items < 2LL * num_sms * 8 && small_items > big_items)
    return scatter_k<16, 1>(p, weights, npad_max, num_sms, s);
  if (v32 && p.rowbytes > 8192) return scatter_k<32, 4>(p, weights, npad_max, num_sms, s);
  if (v32) return scatter_k<32, 2>(p, weights, npad_max, num_sms, s);
  return scatter_k<16, 4>(p, weights, npad_max, num_sms, s);
}

namespace {
template <int KMAX>
cudaError_t scatter_sharded_k(const RowParams& p, bool weights, int npad_max, int num_sms,
                              cudaStream_t s) {
  // 16-byte vectors: the table's addresses are only known to be 16-byte
  // aligned.  4 vectors per lane (2 KB per warp item), 2 from K = 8 up, so that
  // the K destination rows and the loaded vectors stay in registers.
  constexpr int VB = 16, U = KMAX >= 8 ? 2 : 4;
  const long long HV = p.rowbytes / VB;
  const long long cpr = (HV + 32 * U - 1) / (32 * U);
  if (weights)
    return launch_scatter_grid(ep_scatter_rows_kernel<VB, U, KMAX, true, false, true>, p, cpr, npad_max, num_sms, s);
  return launch_scatter_grid(ep_scatter_rows_kernel<VB, U, KMAX, false, false, true>, p, cpr, npad_max, num_sms, s);
}

// Rank-major push: the sharded scatter's vectors, plus the routing rows.
template <int KMAX>
cudaError_t scatter_rank_major_k(const RowParams& p, int num_sms, cudaStream_t s) {
  constexpr int VB = 16, U = KMAX >= 8 ? 2 : 4;
  const long long cpr = (p.rowbytes / VB + 32 * U - 1) / (32 * U);
  return launch_scatter_grid(ep_scatter_rows_kernel<VB, U, KMAX, false, false, true, true>, p, cpr, 0, num_sms, s);
}

template <int DT, int KMAX, int U>
cudaError_t gather_rank_major_k(const RowParams& p, int num_sms, cudaStream_t s) {
  const int HV = p.rowbytes >> 4;
  const long long cpr = (HV + 32 * U - 1) / (32 * U);
  const long long items = static_cast<long long>(p.T) * cpr;
  return launch_rows(ep_gather_sum_kernel<DT, KMAX, U, true, false, true, true>, p, items, num_sms, s, true);
}

// Rank-major dispatch_bwd: the sharded gather-sum's shapes, weight
// gradients from the owners' [rows][K].
template <int DT>
cudaError_t gather_rank_major_dt(const RowParams& p, int num_sms, cudaStream_t s) {
  if (p.K <= 2) return gather_rank_major_k<DT, 2, 2>(p, num_sms, s);
  if (p.K <= 4) return gather_rank_major_k<DT, 4, 4>(p, num_sms, s);
  if (p.K <= 8) return gather_rank_major_k<DT, 8, 2>(p, num_sms, s);
  if (p.K <= 16) return gather_rank_major_k<DT, 16, 1>(p, num_sms, s);
  return gather_rank_major_k<DT, 32, 1>(p, num_sms, s);
}

template <int DT, int KMAX, int U>
cudaError_t gather_sharded_k(const RowParams& p, bool weights, int num_sms, cudaStream_t s) {
  const int HV = p.rowbytes >> 4;
  const long long cpr = (HV + 32 * U - 1) / (32 * U);
  const long long items = static_cast<long long>(p.T) * cpr;
  if (weights) return launch_rows(ep_gather_sum_kernel<DT, KMAX, U, true, false, true>, p, items, num_sms, s, true);
  return launch_rows(ep_gather_sum_kernel<DT, KMAX, U, false, false, true>, p, items, num_sms, s, true);
}

template <int DT>
cudaError_t gather_sharded_dt(const RowParams& p, bool weights, int num_sms, cudaStream_t s) {
  if (p.K <= 2) return gather_sharded_k<DT, 2, 2>(p, weights, num_sms, s);
  if (p.K <= 4) return gather_sharded_k<DT, 4, 4>(p, weights, num_sms, s);
  if (p.K <= 8) return gather_sharded_k<DT, 8, 2>(p, weights, num_sms, s);
  if (p.K <= 16) return gather_sharded_k<DT, 16, 1>(p, weights, num_sms, s);
  return gather_sharded_k<DT, 32, 1>(p, weights, num_sms, s);
}
}  // namespace

cudaError_t launch_scatter_sharded(const RowParams& p, bool weights, int npad_max, int num_sms,
                                   cudaStream_t s) {
  if (p.K <= 2) return scatter_sharded_k<2>(p, weights, npad_max, num_sms, s);
  if (p.K <= 4) return scatter_sharded_k<4>(p, weights, npad_max, num_sms, s);
  if (p.K <= 8) return scatter_sharded_k<8>(p, weights, npad_max, num_sms, s);
  if (p.K <= 16) return scatter_sharded_k<16>(p, weights, npad_max, num_sms, s);
  return scatter_sharded_k<32>(p, weights, npad_max, num_sms, s);
}

cudaError_t launch_gather_sharded(const RowParams& p, bool weights, int num_sms, cudaStream_t s) {
  if (p.dtype == EP_DTYPE_FP16) return gather_sharded_dt<EP_DTYPE_FP16>(p, weights, num_sms, s);
  if (p.dtype == EP_DTYPE_FP32) return gather_sharded_dt<EP_DTYPE_FP32>(p, weights, num_sms, s);
  return gather_sharded_dt<EP_DTYPE_BF16>(p, weights, num_sms, s);
}

cudaError_t launch_gather(const RowParams& p, bool weights, bool scaled, int num_sms,
                          cudaStream_t s) {
  if (p.dtype == EP_DTYPE_FP16) return gather_dt<EP_DTYPE_FP16>(p, weights, scaled, num_sms, s);
  if (p.dtype == EP_DTYPE_FP32) return gather_dt<EP_DTYPE_FP32>(p, weights, scaled, num_sms, s);
  return gather_dt<EP_DTYPE_BF16>(p, weights, scaled, num_sms, s);
}

cudaError_t launch_combine_bwd_scaled(const RowParams& p, int npad_max, int num_sms,
                                      cudaStream_t s) {
  if (p.dtype == EP_DTYPE_FP16) return combine_bwd_scaled_dt<EP_DTYPE_FP16>(p, npad_max, num_sms, s);
  if (p.dtype == EP_DTYPE_FP32) return combine_bwd_scaled_dt<EP_DTYPE_FP32>(p, npad_max, num_sms, s);
  return combine_bwd_scaled_dt<EP_DTYPE_BF16>(p, npad_max, num_sms, s);
}

cudaError_t launch_scatter_rank_major(const RowParams& p, int num_sms, cudaStream_t s) {
  if (p.K <= 2) return scatter_rank_major_k<2>(p, num_sms, s);
  if (p.K <= 4) return scatter_rank_major_k<4>(p, num_sms, s);
  if (p.K <= 8) return scatter_rank_major_k<8>(p, num_sms, s);
  if (p.K <= 16) return scatter_rank_major_k<16>(p, num_sms, s);
  return scatter_rank_major_k<32>(p, num_sms, s);
}

cudaError_t launch_gather_rank_major_bwd(const RowParams& p, int num_sms, cudaStream_t s) {
  if (p.dtype == EP_DTYPE_FP16) return gather_rank_major_dt<EP_DTYPE_FP16>(p, num_sms, s);
  if (p.dtype == EP_DTYPE_FP32) return gather_rank_major_dt<EP_DTYPE_FP32>(p, num_sms, s);
  return gather_rank_major_dt<EP_DTYPE_BF16>(p, num_sms, s);
}

}  // namespace ep
