// ep_api.cu -- the C ABI of libep: registration, host-side validation, launch
// configuration.  No per-step allocation and no host synchronisation except
// in ep_read_info.
//
// Mirrors TransformerEngine PR #3034, "Expert Parallelism: common C API + NCCL
// EP backend": "Lifecycle (host-only, eager)" (nvte_ep_register_layer) and
// "Per-step (allocation-free, CUDA-graph capturable)" (prepare, dispatch,
// combine, dispatch_bwd, combine_bwd).  Return codes replace the throwing C++
// backend; one GPU replaces the communicator.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "ep_internal.cuh"

namespace ep {
cudaError_t probe_kernel_image();
}

namespace {

using ep::LayerInfo;
using ep::Layout;

constexpr uint64_t kMaxLayers = 1u << 16;
constexpr int kMaxDevices = 64;
constexpr long long kMaxRoutes = 1LL << 24;
constexpr long long kMaxChunks = 4096;

LayerInfo* g_layers[kMaxLayers];
std::atomic<uint64_t> g_num_layers{0};
std::mutex g_register_mu;
std::atomic<uint64_t> g_launches{0};

thread_local std::string g_error;

struct DeviceInfo {
  std::atomic<int> state{0};  // 0 unknown, 1 supported, 2 unsupported
  int num_sms = 0;
  int max_cluster = ep::kMaxCluster;  // largest cluster of the one-launch prepare
  int max_cluster_shard = ep::kMaxCluster;  // and of the sharded routing modes
  int wide_ctas = 0;  // CTAs of the grid-wide prepare that fit at once (0: not used)
};
DeviceInfo g_devices[kMaxDevices];
std::mutex g_device_mu;

ep_status_t fail(ep_status_t code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_error = buf;
  return code;
}

ep_status_t cuda_fail(cudaError_t e, const char* where) {
  return fail(EP_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

// The current device must be compute capability 10.3 (GB300) and able to load
// this library's kernels.  Checked once per device.
ep_status_t check_device(int* num_sms, int* max_cluster = nullptr, int* max_cluster_shard = nullptr,
                         int* wide_ctas = nullptr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(EP_ERR_LIMIT, "device ordinal %d out of range", dev);
  DeviceInfo& d = g_devices[dev];
  int st = d.state.load(std::memory_order_acquire);
  if (st == 0) {
    std::lock_guard<std::mutex> lock(g_device_mu);
    st = d.state.load(std::memory_order_relaxed);
    if (st == 0) {
      int major = 0, minor = 0, sms = 0;
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
      bool ok = (major == 10 && minor == 3) && ep::probe_kernel_image() == cudaSuccess;
      cudaGetLastError();
      d.num_sms = sms > 0 ? sms : 1;
      if (ok) {
        d.max_cluster = ep::prepare_max_cluster();
        d.max_cluster_shard = ep::shard_max_cluster();
        d.wide_ctas = ep::prepare_wide_ctas();
      }
      st = ok ? 1 : 2;
      d.state.store(st, std::memory_order_release);
      if (!ok) g_error = "device is not sm_103 (GB300) or cannot load libep kernels";
    }
  }
  if (st != 1) return fail(EP_ERR_UNSUPPORTED_ARCH, "device %d is not compute capability 10.3 (GB300), or the sm_103a kernels do not load", dev);
  *num_sms = d.num_sms;
  if (max_cluster != nullptr) *max_cluster = d.max_cluster;
  if (max_cluster_shard != nullptr) *max_cluster_shard = d.max_cluster_shard;
  if (wide_ctas != nullptr) *wide_ctas = d.wide_ctas;
  return EP_OK;
}

// A sharded layer's batch must fit the routing map's cluster on this device.
ep_status_t check_shard_routes(const LayerInfo* L, int64_t T, int max_cluster_shard) {
  const int E = static_cast<int>(L->cfg.num_experts);
  const long long lim = ep::shard_max_routes(E, max_cluster_shard);
  if (T * L->cfg.top_k > lim)
    return fail(EP_ERR_LIMIT, "%lld routes exceed the %lld a sharded layer's routing map takes at %d experts on this device",
                (long long)(T * L->cfg.top_k), lim, E);
  return EP_OK;
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

Layout make_layout(const ep_layer_config_t& c, int64_t R, int64_t nranks) {
  Layout L;
  const int64_t E = c.num_experts, K = c.top_k, routes = c.max_tokens * K;
  const int64_t Eown = nranks > 0 ? E / nranks : E;  // experts whose rows this rank holds
  size_t off = ep::kHeaderBytes;
  L.counts = off;
  off = align256(off + static_cast<size_t>(E) * 4);
  L.offsets = off;
  off = align256(off + static_cast<size_t>(E + 1) * 4);
  L.slot = off;
  off = align256(off + static_cast<size_t>(routes > 0 ? routes : 1) * 4);
  int64_t pad = Eown * (c.max_alignment - 1);
  if (pad > R) pad = R;
  if (pad < 1) pad = 1;
  L.pad_cap = pad;
  L.pad_list = off;
  off = align256(off + static_cast<size_t>(pad) * 4);
  const int64_t per_chunk = static_cast<int64_t>(ep::chunk_warps(static_cast<int>(E))) * 32;
  int64_t chunks = (routes + per_chunk - 1) / per_chunk;
  if (chunks < 1) chunks = 1;
  if (chunks > kMaxChunks) chunks = kMaxChunks;
  L.max_chunks = chunks;
  L.hist = off;  // [E][chunks] for the chunked prepare, [chunks][E rounded up to 4] grid-wide
  off = align256(off + static_cast<size_t>((E + 3) & ~int64_t{3}) * chunks * 4);
  L.badflag = off;
  off = align256(off + static_cast<size_t>(chunks) * 4);
  L.dest = off;
  if (nranks > 0) off = align256(off + static_cast<size_t>(routes > 0 ? routes : 1) * 4);
  L.oidx = L.owner = 0;
  L.total = off;
  return L;
}

// A rank-major layer routes its tokens over N pseudo-experts (one per owner
// rank, alignment 1), and keeps beside the maps the per-route owner ids the
// routing reads and every route's owner.
Layout make_rank_major_layout(const ep_layer_config_t& c, int64_t R, int64_t nranks) {
  ep_layer_config_t r = c;
  r.num_experts = nranks;
  r.max_alignment = 1;
  Layout L = make_layout(r, R, nranks);
  const size_t routes = static_cast<size_t>(c.max_tokens * c.top_k > 0 ? c.max_tokens * c.top_k : 1);
  size_t off = L.total;
  L.oidx = off;
  off = align256(off + routes * 8);
  L.owner = off;
  off = align256(off + routes * 4);
  L.total = off;
  return L;
}

// kind: 0 a single-buffer call, 1 a sharded call, 2 any layer, 3 a rank-major call.
ep_status_t lookup(const ep_handle_t& h, const LayerInfo** out, int kind = 0) {
  const uint64_t n = g_num_layers.load(std::memory_order_acquire);
  if (h.id == 0 || h.id > n) return fail(EP_ERR_NOT_REGISTERED, "layer id %llu is not registered", (unsigned long long)h.id);
  if (h.mem == nullptr) return fail(EP_ERR_INVALID_ARG, "handle memory is NULL");
  if (reinterpret_cast<uintptr_t>(h.mem) % 256 != 0) return fail(EP_ERR_INVALID_ARG, "handle memory is not 256-byte aligned");
  const LayerInfo* L = g_layers[h.id - 1];
  if (kind == 0 && L->nranks > 0)
    return fail(EP_ERR_INVALID_ARG, "layer %llu is sharded: use the ep_shard_* calls", (unsigned long long)h.id);
  if (kind == 1 && (L->nranks == 0 || L->rank_major))
    return fail(EP_ERR_INVALID_ARG, "layer %llu is not an expert-major sharded layer (ep_register_layer_sharded)", (unsigned long long)h.id);
  if (kind == 3 && !L->rank_major)
    return fail(EP_ERR_INVALID_ARG, "layer %llu is not a rank-major layer (ep_register_layer_rank_major)", (unsigned long long)h.id);
  *out = L;
  return EP_OK;
}

bool misaligned(const void* p, size_t a) { return reinterpret_cast<uintptr_t>(p) % a != 0; }

// log2(A) when A is a power of two, else -1.
int log2_if_pow2(int64_t A) {
  if (A < 1 || (A & (A - 1)) != 0) return -1;
  int k = 0;
  while ((int64_t{1} << k) < A) ++k;
  return k;
}

ep_status_t check_tokens(const LayerInfo* L, int64_t T) {
  if (T < 0 || T > L->cfg.max_tokens)
    return fail(EP_ERR_SHAPE, "num_tokens %lld outside [0, max_tokens=%lld]", (long long)T, (long long)L->cfg.max_tokens);
  return EP_OK;
}

ep_status_t check_payload(const void* p, int64_t T, const char* name, bool needed) {
  if (!needed) return EP_OK;
  if (p == nullptr) return fail(EP_ERR_INVALID_ARG, "%s is NULL", name);
  if (misaligned(p, 16)) return fail(EP_ERR_INVALID_ARG, "%s is not 16-byte aligned", name);
  (void)T;
  return EP_OK;
}

ep_status_t check_f32(const void* p, const char* name, bool needed) {
  if (!needed) return EP_OK;
  if (p == nullptr) return fail(EP_ERR_INVALID_ARG, "%s is NULL", name);
  if (misaligned(p, 4)) return fail(EP_ERR_INVALID_ARG, "%s is not 4-byte aligned", name);
  return EP_OK;
}

template <typename T>
T* at(void* mem, size_t off) { return reinterpret_cast<T*>(static_cast<char*>(mem) + off); }

ep::RowParams row_params(const LayerInfo* L, const ep_handle_t& h, int64_t T) {
  ep::RowParams p;
  p.hdr = at<int>(h.mem, 0);
  p.slot = at<int>(h.mem, L->lay.slot);
  p.pad_list = at<int>(h.mem, L->lay.pad_list);
  p.T = static_cast<int>(T);
  p.K = static_cast<int>(L->cfg.top_k);
  p.H = static_cast<int>(L->cfg.hidden);
  p.R = static_cast<int>(L->R);
  p.pad_cap = static_cast<int>(L->lay.pad_cap);
  p.dtype = static_cast<int>(L->cfg.dtype);
  p.rowbytes = static_cast<int>(L->cfg.hidden * L->es);
  p.src = nullptr;
  p.dst = nullptr;
  p.w_in = nullptr;
  p.w_out = nullptr;
  p.scale = nullptr;
  p.aux = nullptr;
  p.prefetch = 0;
  p.resident_warps = 0;  // set at launch
  p.tok_warps = 0;       // set at launch (scatter)
  p.dest = at<int>(h.mem, L->lay.dest);
  p.nranks = static_cast<int>(L->nranks);
  p.rank = static_cast<int>(L->rank);
  p.dst_tab = nullptr;
  p.src_tab = nullptr;
  p.wout_tab = nullptr;
  p.win_tab = nullptr;
  p.idx = nullptr;
  p.owner = nullptr;
  p.idx_tab = nullptr;
  p.eloc = 0;
  return p;
}

// Routing-map parameters of a prepare on handle h (sharded fields unset).
ep::RouteParams route_params(const LayerInfo* L, const ep_handle_t& h, const int64_t* topk_idx,
                             int64_t T, int32_t* token_counts, int64_t A) {
  ep::RouteParams p;
  p.idx = reinterpret_cast<const long long*>(topk_idx);
  p.n = static_cast<int>(T * L->cfg.top_k);
  p.T = static_cast<int>(T);
  p.K = static_cast<int>(L->cfg.top_k);
  p.E = static_cast<int>(L->cfg.num_experts);
  p.A = static_cast<int>(A);
  p.a_log2 = log2_if_pow2(A);
  p.R = L->R;
  p.pad_cap = L->lay.pad_cap;
  p.warps = 0;
  p.chunk = 0;
  p.nchunks = static_cast<int>(L->lay.max_chunks);
  p.hdr = at<int>(h.mem, 0);
  p.counts = at<int>(h.mem, L->lay.counts);
  p.counts_user = token_counts;
  p.offsets = at<int>(h.mem, L->lay.offsets);
  p.slot = at<int>(h.mem, L->lay.slot);
  p.pad_list = at<int>(h.mem, L->lay.pad_list);
  p.hist = at<int>(h.mem, L->lay.hist);
  p.badflag = at<int>(h.mem, L->lay.badflag);
  p.all_counts = nullptr;
  p.nranks = static_cast<int>(L->nranks);
  p.rank = static_cast<int>(L->rank);
  p.dest = at<int>(h.mem, L->lay.dest);
  p.idx_in = nullptr;
  p.oidx = nullptr;
  p.owner = nullptr;
  p.E_all = p.E;
  p.eloc = 0;
  return p;
}

// A device table of N addresses (sharded row calls): present and 8-byte aligned.
ep_status_t check_table(const void* tab, const char* name) {
  if (tab == nullptr) return fail(EP_ERR_INVALID_ARG, "%s (table of per-rank addresses) is NULL", name);
  if (misaligned(tab, 8)) return fail(EP_ERR_INVALID_ARG, "%s (table of per-rank addresses) is not 8-byte aligned", name);
  return EP_OK;
}

ep_status_t register_layer(ep_layer_config_t c, int64_t nranks, int64_t rank, uint64_t* id,
                           size_t* handle_mem_size) {
  if (id == nullptr || handle_mem_size == nullptr) return fail(EP_ERR_INVALID_ARG, "id and handle_mem_size must not be NULL");
  if (c.num_experts < 1 || c.num_experts > EP_MAX_EXPERTS)
    return fail(EP_ERR_LIMIT, "num_experts %lld outside [1, %d]", (long long)c.num_experts, EP_MAX_EXPERTS);
  if (c.top_k < 1 || c.top_k > EP_MAX_TOPK)
    return fail(EP_ERR_LIMIT, "top_k %lld outside [1, %d]", (long long)c.top_k, EP_MAX_TOPK);
  if (c.hidden < 8 || c.hidden % 8 != 0 || c.hidden > (1 << 20))
    return fail(EP_ERR_LIMIT, "hidden %lld must be a positive multiple of 8 (16-byte rows), at most 2^20", (long long)c.hidden);
  if (c.max_tokens < 0 || c.max_tokens * c.top_k > kMaxRoutes)
    return fail(EP_ERR_LIMIT, "max_tokens*top_k must lie in [0, 2^24]");
  if (c.max_alignment < 1 || c.max_alignment > (1 << 20))
    return fail(EP_ERR_LIMIT, "max_alignment %lld outside [1, 2^20]", (long long)c.max_alignment);
  const int64_t routes = c.max_tokens * c.top_k;
  if (nranks > 0) {
    if (c.num_experts % nranks != 0)
      return fail(EP_ERR_INVALID_ARG, "num_ranks %lld must divide num_experts %lld", (long long)nranks, (long long)c.num_experts);
    const long long lim = ep::shard_max_routes(static_cast<int>(c.num_experts), ep::kMaxClusterWide);
    if (routes > lim)
      return fail(EP_ERR_LIMIT, "sharded layers take at most %lld routes (max_tokens*top_k) per rank at %lld experts",
                  lim, (long long)c.num_experts);
  }
  // Rows an owner may receive: every rank's routes to its experts.
  const int64_t in_routes = nranks > 0 ? nranks * routes : routes;
  const int64_t own = nranks > 0 ? c.num_experts / nranks : c.num_experts;
  const int64_t worst = in_routes + (own < in_routes ? own : in_routes) * (c.max_alignment - 1);
  if (in_routes + own * (c.max_alignment - 1) >= (1LL << 31))
    return fail(EP_ERR_LIMIT, "max_tokens*top_k (times num_ranks) + experts*(max_alignment-1) must stay below 2^31");
  if (c.recv_capacity < 0) return fail(EP_ERR_INVALID_ARG, "recv_capacity must be >= 0");
  if (c.dtype != EP_DTYPE_BF16 && c.dtype != EP_DTYPE_FP16 && c.dtype != EP_DTYPE_FP32)
    return fail(EP_ERR_INVALID_ARG, "dtype %lld is not an ep_dtype_t", (long long)c.dtype);
  const int es = c.dtype == EP_DTYPE_FP32 ? 4 : 2;
  const int64_t R = c.recv_capacity == 0 ? worst : c.recv_capacity;
  if (R >= (1LL << 31)) return fail(EP_ERR_LIMIT, "recv_capacity must stay below 2^31 rows");
  const int64_t cpr = (c.hidden * es / 16 + 31) / 32;
  const int64_t pad = own * (c.max_alignment - 1) < R ? own * (c.max_alignment - 1) : R;
  if ((c.max_tokens + pad) * cpr >= (1LL << 31))
    return fail(EP_ERR_LIMIT, "(max_tokens + padding rows) * row chunks must stay below 2^31");

  LayerInfo* info = new LayerInfo;
  info->cfg = c;
  info->R = R;
  info->es = es;
  info->lay = make_layout(c, R, nranks);
  info->nranks = nranks;
  info->rank = rank;
  info->rank_major = false;
  std::lock_guard<std::mutex> lock(g_register_mu);
  const uint64_t n = g_num_layers.load(std::memory_order_relaxed);
  if (n >= kMaxLayers) {
    delete info;
    return fail(EP_ERR_LIMIT, "too many layers registered (%llu)", (unsigned long long)kMaxLayers);
  }
  g_layers[n] = info;
  g_num_layers.store(n + 1, std::memory_order_release);
  *id = n + 1;
  *handle_mem_size = info->lay.total;
  return EP_OK;
}

// Publishes a registered layer; fails when the table is full.
ep_status_t publish(LayerInfo* info, uint64_t* id, size_t* handle_mem_size) {
  std::lock_guard<std::mutex> lock(g_register_mu);
  const uint64_t n = g_num_layers.load(std::memory_order_relaxed);
  if (n >= kMaxLayers) {
    delete info;
    return fail(EP_ERR_LIMIT, "too many layers registered (%llu)", (unsigned long long)kMaxLayers);
  }
  g_layers[n] = info;
  g_num_layers.store(n + 1, std::memory_order_release);
  *id = n + 1;
  *handle_mem_size = info->lay.total;
  return EP_OK;
}

ep_status_t register_rank_major(ep_layer_config_t c, int64_t nranks, int64_t rank, uint64_t* id,
                                size_t* handle_mem_size) {
  if (id == nullptr || handle_mem_size == nullptr) return fail(EP_ERR_INVALID_ARG, "id and handle_mem_size must not be NULL");
  if (nranks < 1 || nranks > EP_MAX_RANKS)
    return fail(EP_ERR_LIMIT, "num_ranks %lld outside [1, %d]", (long long)nranks, EP_MAX_RANKS);
  if (rank < 0 || rank >= nranks)
    return fail(EP_ERR_INVALID_ARG, "rank %lld outside [0, num_ranks=%lld)", (long long)rank, (long long)nranks);
  if (c.num_experts < 1 || c.num_experts > EP_MAX_EXPERTS)
    return fail(EP_ERR_LIMIT, "num_experts %lld outside [1, %d]", (long long)c.num_experts, EP_MAX_EXPERTS);
  if (c.num_experts % nranks != 0)
    return fail(EP_ERR_INVALID_ARG, "num_ranks %lld must divide num_experts %lld", (long long)nranks, (long long)c.num_experts);
  if (c.top_k < 1 || c.top_k > EP_MAX_TOPK)
    return fail(EP_ERR_LIMIT, "top_k %lld outside [1, %d]", (long long)c.top_k, EP_MAX_TOPK);
  if (c.hidden < 8 || c.hidden % 8 != 0 || c.hidden > (1 << 20))
    return fail(EP_ERR_LIMIT, "hidden %lld must be a positive multiple of 8 (16-byte rows), at most 2^20", (long long)c.hidden);
  const long long lim = ep::shard_max_routes(static_cast<int>(nranks), ep::kMaxClusterWide);
  if (c.max_tokens < 0 || c.max_tokens * c.top_k > lim)
    return fail(EP_ERR_LIMIT, "rank-major layers take at most %lld routes (max_tokens*top_k) per rank at %lld ranks",
                lim, (long long)nranks);
  if (c.recv_capacity < 0) return fail(EP_ERR_INVALID_ARG, "recv_capacity must be >= 0");
  if (c.dtype != EP_DTYPE_BF16 && c.dtype != EP_DTYPE_FP16 && c.dtype != EP_DTYPE_FP32)
    return fail(EP_ERR_INVALID_ARG, "dtype %lld is not an ep_dtype_t", (long long)c.dtype);
  // A token goes at most once to each owner: N * max_tokens rows at worst.
  const int64_t R = c.recv_capacity == 0 ? nranks * c.max_tokens : c.recv_capacity;
  if (R >= (1LL << 31)) return fail(EP_ERR_LIMIT, "recv_capacity must stay below 2^31 rows");
  const int es = c.dtype == EP_DTYPE_FP32 ? 4 : 2;
  LayerInfo* info = new LayerInfo;
  info->cfg = c;
  info->R = R;
  info->es = es;
  info->lay = make_rank_major_layout(c, R, nranks);
  info->nranks = nranks;
  info->rank = rank;
  info->rank_major = true;
  return publish(info, id, handle_mem_size);
}

// Routing-map parameters of a rank-major count or prepare: the routing reads
// the per-route owner ids (N pseudo-experts, alignment 1) that the owners
// kernel writes from topk_idx just before.
ep::RouteParams rank_major_route_params(const LayerInfo* L, const ep_handle_t& h, const int64_t* topk_idx,
                                        int64_t T, int32_t* counts_user) {
  ep::RouteParams p;
  const int N = static_cast<int>(L->nranks);
  p.idx = at<const long long>(h.mem, L->lay.oidx);
  p.n = static_cast<int>(T * L->cfg.top_k);
  p.T = static_cast<int>(T);
  p.K = static_cast<int>(L->cfg.top_k);
  p.E = N;
  p.A = 1;
  p.a_log2 = 0;
  p.R = L->R;
  p.pad_cap = L->lay.pad_cap;
  p.warps = 0;
  p.chunk = 0;
  p.nchunks = static_cast<int>(L->lay.max_chunks);
  p.hdr = at<int>(h.mem, 0);
  p.counts = at<int>(h.mem, L->lay.counts);
  p.counts_user = counts_user;
  p.offsets = at<int>(h.mem, L->lay.offsets);
  p.slot = at<int>(h.mem, L->lay.slot);
  p.pad_list = at<int>(h.mem, L->lay.pad_list);
  p.hist = at<int>(h.mem, L->lay.hist);
  p.badflag = at<int>(h.mem, L->lay.badflag);
  p.all_counts = nullptr;
  p.nranks = N;
  p.rank = static_cast<int>(L->rank);
  p.dest = at<int>(h.mem, L->lay.dest);
  p.idx_in = reinterpret_cast<const long long*>(topk_idx);
  p.oidx = at<long long>(h.mem, L->lay.oidx);
  p.owner = at<int>(h.mem, L->lay.owner);
  p.E_all = static_cast<int>(L->cfg.num_experts);
  p.eloc = static_cast<int>(L->cfg.num_experts / N);
  return p;
}

// Row-kernel parameters of a rank-major row call (no padding rows).
ep::RowParams rank_major_row_params(const LayerInfo* L, const ep_handle_t& h, int64_t T) {
  ep::RowParams p = row_params(L, h, T);
  p.owner = at<int>(h.mem, L->lay.owner);
  p.eloc = static_cast<int>(L->cfg.num_experts / L->nranks);
  return p;
}

}  // namespace

extern "C" {

uint32_t ep_abi_version(void) { return EP_ABI_VERSION; }

const char* ep_last_error(void) { return g_error.c_str(); }

uint64_t ep_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

ep_status_t ep_register_layer(ep_layer_config_t c, uint64_t* id, size_t* handle_mem_size) {
  return register_layer(c, 0, 0, id, handle_mem_size);
}

ep_status_t ep_register_layer_sharded(ep_layer_config_t c, int64_t num_ranks, int64_t rank,
                                      uint64_t* id, size_t* handle_mem_size) {
  if (num_ranks < 1 || num_ranks > EP_MAX_RANKS)
    return fail(EP_ERR_LIMIT, "num_ranks %lld outside [1, %d]", (long long)num_ranks, EP_MAX_RANKS);
  if (rank < 0 || rank >= num_ranks)
    return fail(EP_ERR_INVALID_ARG, "rank %lld outside [0, num_ranks=%lld)", (long long)rank, (long long)num_ranks);
  return register_layer(c, num_ranks, rank, id, handle_mem_size);
}
ep_status_t ep_recv_capacity(uint64_t id, int64_t* rows) {
  if (rows == nullptr) return fail(EP_ERR_INVALID_ARG, "rows is NULL");
  const uint64_t n = g_num_layers.load(std::memory_order_acquire);
  if (id == 0 || id > n) return fail(EP_ERR_NOT_REGISTERED, "layer id %llu is not registered", (unsigned long long)id);
  *rows = g_layers[id - 1]->R;
  return EP_OK;
}

ep_status_t ep_prepare(ep_handle_t h, const int64_t* topk_idx, int64_t T, int32_t* token_counts,
                       int64_t alignment, void* stream) {
  const LayerInfo* L = nullptr;
  ep_status_t st = lookup(h, &L);
  if (st != EP_OK) return st;
  if ((st = check_tokens(L, T)) != EP_OK) return st;
  if (T > 0 && topk_idx == nullptr) return fail(EP_ERR_INVALID_ARG, "topk_idx is NULL");
  if (topk_idx != nullptr && misaligned(topk_idx, 8)) return fail(EP_ERR_INVALID_ARG, "topk_idx is not 8-byte aligned");
  if (token_counts == nullptr) return fail(EP_ERR_INVALID_ARG, "token_counts is NULL");
  if (misaligned(token_counts, 4)) return fail(EP_ERR_INVALID_ARG, "token_counts is not 4-byte aligned");
  if (alignment < 1 || alignment > L->cfg.max_alignment)
    return fail(EP_ERR_SHAPE, "alignment %lld outside [1, max_alignment=%lld]", (long long)alignment, (long long)L->cfg.max_alignment);
  int sms = 0, max_cluster = 0, wide_ctas = 0;
  if ((st = check_device(&sms, &max_cluster, nullptr, &wide_ctas)) != EP_OK) return st;

  ep::RouteParams p;
  p.idx = reinterpret_cast<const long long*>(topk_idx);
  p.n = static_cast<int>(T * L->cfg.top_k);
  p.T = static_cast<int>(T);
  p.K = static_cast<int>(L->cfg.top_k);
  p.E = static_cast<int>(L->cfg.num_experts);
  p.A = static_cast<int>(alignment);
  p.a_log2 = log2_if_pow2(alignment);
  p.R = L->R;
  p.pad_cap = L->lay.pad_cap;
  p.warps = 0;
  p.chunk = 0;
  p.nchunks = static_cast<int>(L->lay.max_chunks);
  p.hdr = at<int>(h.mem, 0);
  p.counts = at<int>(h.mem, L->lay.counts);
  p.counts_user = token_counts;
  p.offsets = at<int>(h.mem, L->lay.offsets);
  p.slot = at<int>(h.mem, L->lay.slot);
  p.pad_list = at<int>(h.mem, L->lay.pad_list);
  p.hist = at<int>(h.mem, L->lay.hist);
  p.badflag = at<int>(h.mem, L->lay.badflag);
  p.all_counts = nullptr;
  p.nranks = 0;
  p.rank = 0;
  p.dest = nullptr;
  int launched = 0;
  cudaError_t e = ep::launch_prepare(p, sms, max_cluster, wide_ctas, static_cast<cudaStream_t>(stream),
                                     &launched);
  g_launches.fetch_add(launched, std::memory_order_relaxed);
  if (e != cudaSuccess) return cuda_fail(e, "ep_prepare launch");
  return EP_OK;
}

// Same routing map as ep_prepare, built with the per-chunk counters in
// libep's fixed device array instead of the scratch part of handle memory.
// Allocates nothing.  The first call on a device looks up the array's device
// address (cudaGetSymbolAddress), so make that first call before any stream
// capture on that device.
ep_status_t ep_prepare_static_scratch(ep_handle_t h, const int64_t* topk_idx, int64_t T,
                                      int32_t* token_counts, int64_t alignment, void* stream) {
  const LayerInfo* L = nullptr;
  ep_status_t st = lookup(h, &L);
  if (st != EP_OK) return st;
  if ((st = check_tokens(L, T)) != EP_OK) return st;
  if (T > 0 && topk_idx == nullptr) return fail(EP_ERR_INVALID_ARG, "topk_idx is NULL");
  if (topk_idx != nullptr && misaligned(topk_idx, 8)) return fail(EP_ERR_INVALID_ARG, "topk_idx is not 8-byte aligned");
  if (token_counts == nullptr) return fail(EP_ERR_INVALID_ARG, "token_counts is NULL");
  if (misaligned(token_counts, 4)) return fail(EP_ERR_INVALID_ARG, "token_counts is not 4-byte aligned");
  if (alignment < 1 || alignment > L->cfg.max_alignment)
    return fail(EP_ERR_SHAPE, "alignment %lld outside [1, max_alignment=%lld]", (long long)alignment, (long long)L->cfg.max_alignment);
  int sms = 0;
  if ((st = check_device(&sms)) != EP_OK) return st;
  const int n = static_cast<int>(T * L->cfg.top_k);
  const int E = static_cast<int>(L->cfg.num_experts);
  int w = 0, chunk = 0, nchunks = 0;
  if (!ep::static_scratch_plan(n, E, sms, &w, &chunk, &nchunks))
    return fail(EP_ERR_LIMIT,
                "%d routes over %d experts do not fit the fixed scratch array of %d ints "
                "(needs (experts+1) x chunks counters, chunks of at most %d routes); use ep_prepare",
                n, E, ep::kStaticScratchInts, ep::chunk_warps(E) * 32 * ep::kMaxJ);
  int* scratch = nullptr;
  cudaError_t e = ep::static_scratch_address(&scratch);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress of the fixed scratch array");

  ep::RouteParams p;
  p.idx = reinterpret_cast<const long long*>(topk_idx);
  p.n = n;
  p.T = static_cast<int>(T);
  p.K = static_cast<int>(L->cfg.top_k);
  p.E = E;
  p.A = static_cast<int>(alignment);
  p.a_log2 = log2_if_pow2(alignment);
  p.R = L->R;
  p.pad_cap = L->lay.pad_cap;
  p.warps = 0;
  p.chunk = 0;
  p.nchunks = 0;
  p.hdr = at<int>(h.mem, 0);
  p.counts = at<int>(h.mem, L->lay.counts);
  p.counts_user = token_counts;
  p.offsets = at<int>(h.mem, L->lay.offsets);
  p.slot = at<int>(h.mem, L->lay.slot);
  p.pad_list = at<int>(h.mem, L->lay.pad_list);
  p.hist = nullptr;
  p.badflag = nullptr;
  p.all_counts = nullptr;
  p.nranks = 0;
  p.rank = 0;
  p.dest = nullptr;
  int launched = 0;
  e = ep::launch_prepare_static_scratch(p, scratch, sms, static_cast<cudaStream_t>(stream), &launched);
  g_launches.fetch_add(launched, std::memory_order_relaxed);
  if (e != cudaSuccess) return cuda_fail(e, "ep_prepare_static_scratch launch");
  return EP_OK;
}

ep_status_t ep_dispatch(ep_handle_t h, const int64_t* topk_idx, int64_t T, const void* tokens,
                        const float* topk_weights, void* recv_tokens, float* recv_topk_weights,
                        void* stream) {
  const LayerInfo* L = nullptr;
  ep_status_t st = lookup(h, &L);
  if (st != EP_OK) return st;
  if ((st = check_tokens(L, T)) != EP_OK) return st;
  if (T > 0 && topk_idx == nullptr) return fail(EP_ERR_INVALID_ARG, "topk_idx is NULL");
  if ((st = check_payload(tokens, T, "tokens", T > 0)) != EP_OK) return st;
  if ((st = check_f32(topk_weights, "topk_weights", T > 0)) != EP_OK) return st;
  if ((st = check_payload(recv_tokens, T, "recv_tokens", true)) != EP_OK) return st;
  if ((st = check_f32(recv_topk_weights, "recv_topk_weights", true)) != EP_OK) return st;
  int sms = 0, max_cluster = 0;
  if ((st = check_device(&sms, &max_cluster)) != EP_OK) return st;
  ep::RowParams p = row_params(L, h, T);
  p.src = tokens;
  p.dst = recv_tokens;
  p.w_in = topk_weights;
  p.w_out = recv_topk_weights;
  // Dispatch normally follows prepare on the stream.  When that prepare is
  // the single cluster launch, most SMs idle while it runs and the token rows
  // can be pulled into L2 meanwhile.  The chunked prepare kernels spread over
  // the SMs, and behind them the prefetch measured no gain.
  p.prefetch = ep::prepare_is_one_launch(T * L->cfg.top_k, static_cast<int>(L->cfg.num_experts),
                                         max_cluster) ? 1 : 0;
  cudaError_t e = ep::launch_scatter(p, true, static_cast<int>(L->lay.pad_cap), sms, static_cast<cudaStream_t>(stream));
  g_launches.fetch_add(1, std::memory_order_relaxed);
  if (e != cudaSuccess) return cuda_fail(e, "ep_dispatch launch");
  return EP_OK;
}

ep_status_t ep_combine(ep_handle_t h, const void* expert_out, int64_t T, void* result,
                       void* stream) {
  const LayerInfo* L = nullptr;
  ep_status_t st = lookup(h, &L);
  if (st != EP_OK) return st;
  if ((st = check_tokens(L, T)) != EP_OK) return st;
  if ((st = check_payload(expert_out, T, "expert_out", true)) != EP_OK) return st;
  if ((st = check_payload(result, T, "result", T > 0)) != EP_OK) return st;
  int sms = 0;
  if ((st = check_device(&sms)) != EP_OK) return st;
  ep::RowParams p = row_params(L, h, T);
  p.src = expert_out;
  p.dst = result;
  cudaError_t e = ep::launch_gather(p, false, false, sms, static_cast<cudaStream_t>(stream));
  g_launches.fetch_add(1, std::memory_order_relaxed);
  if (e != cudaSuccess) return cuda_fail(e, "ep_combine launch");
  return EP_OK;
}

ep_status_t ep_dispatch_bwd(ep_handle_t h, const void* grad, const float* g_recv_topk_weights,
                            int64_t T, void* grad_tokens, float* grad_topk_weights,
                            void* stream) {
  const LayerInfo* L = nullptr;
  ep_status_t st = lookup(h, &L);
  if (st != EP_OK) return st;
  if ((st = check_tokens(L, T)) != EP_OK) return st;
  if ((st = check_payload(grad, T, "grad", true)) != EP_OK) return st;
  if (g_recv_topk_weights != nullptr && misaligned(g_recv_topk_weights, 4))
    return fail(EP_ERR_INVALID_ARG, "g_recv_topk_weights is not 4-byte aligned");
  if ((st = check_payload(grad_tokens, T, "grad_tokens", T > 0)) != EP_OK) return st;
  if ((st = check_f32(grad_topk_weights, "grad_topk_weights", T > 0)) != EP_OK) return st;
  int sms = 0;
  if ((st = check_device(&sms)) != EP_OK) return st;
  ep::RowParams p = row_params(L, h, T);
  p.src = grad;
  p.dst = grad_tokens;
  p.w_in = g_recv_topk_weights;
  p.w_out = grad_topk_weights;
  cudaError_t e = ep::launch_gather(p, true, false, sms, static_cast<cudaStream_t>(stream));
  g_launches.fetch_add(1, std::memory_order_relaxed);
  if (e != cudaSuccess) return cuda_fail(e, "ep_dispatch_bwd launch");
  return EP_OK;
}

ep_status_t ep_combine_bwd(ep_handle_t h, const void* grad, int64_t T, void* grad_expert_out,
                           void* stream) {
  const LayerInfo* L = nullptr;
  ep_status_t st = lookup(h, &L);
  if (st != EP_OK) return st;
  if ((st = check_tokens(L, T)) != EP_OK) return st;
  if ((st = check_payload(grad, T, "grad", T > 0)) != EP_OK) return st;
  if ((st = check_payload(grad_expert_out, T, "grad_expert_out", true)) != EP_OK) return st;
  int sms = 0;
  if ((st = check_device(&sms)) != EP_OK) return st;
  ep::RowParams p = row_params(L, h, T);
  p.src = grad;
  p.dst = grad_expert_out;
  cudaError_t e = ep::launch_scatter(p, false, static_cast<int>(L->lay.pad_cap), sms, static_cast<cudaStream_t>(stream));
  g_launches.fetch_add(1, std::memory_order_relaxed);
  if (e != cudaSuccess) return cuda_fail(e, "ep_combine_bwd launch");
  return EP_OK;
}

ep_status_t ep_combine_weighted(ep_handle_t h, const void* expert_out,
                                const float* recv_topk_weights, int64_t T, void* result,
                                void* stream) {
  const LayerInfo* L = nullptr;
  ep_status_t st = lookup(h, &L);
  if (st != EP_OK) return st;
  if ((st = check_tokens(L, T)) != EP_OK) return st;
  if ((st = check_payload(expert_out, T, "expert_out", true)) != EP_OK) return st;
  if ((st = check_f32(recv_topk_weights, "recv_topk_weights", true)) != EP_OK) return st;
  if ((st = check_payload(result, T, "result", T > 0)) != EP_OK) return st;
  int sms = 0;
  if ((st = check_device(&sms)) != EP_OK) return st;
  ep::RowParams p = row_params(L, h, T);
  p.src = expert_out;
  p.dst = result;
  p.scale = recv_topk_weights;
  cudaError_t e = ep::launch_gather(p, false, true, sms, static_cast<cudaStream_t>(stream));
  g_launches.fetch_add(1, std::memory_order_relaxed);
  if (e != cudaSuccess) return cuda_fail(e, "ep_combine_weighted launch");
  return EP_OK;
}

ep_status_t ep_combine_weighted_bwd(ep_handle_t h, const void* grad, const void* expert_out,
                                    const float* recv_topk_weights, int64_t T,
                                    void* grad_expert_out, float* g_recv_topk_weights,
                                    void* stream) {
  const LayerInfo* L = nullptr;
  ep_status_t st = lookup(h, &L);
  if (st != EP_OK) return st;
  if ((st = check_tokens(L, T)) != EP_OK) return st;
  if ((st = check_payload(grad, T, "grad", T > 0)) != EP_OK) return st;
  if ((st = check_payload(expert_out, T, "expert_out", true)) != EP_OK) return st;
  if ((st = check_f32(recv_topk_weights, "recv_topk_weights", true)) != EP_OK) return st;
  if ((st = check_payload(grad_expert_out, T, "grad_expert_out", true)) != EP_OK) return st;
  if ((st = check_f32(g_recv_topk_weights, "g_recv_topk_weights", true)) != EP_OK) return st;
  int sms = 0;
  if ((st = check_device(&sms)) != EP_OK) return st;
  ep::RowParams p = row_params(L, h, T);
  p.src = grad;
  p.dst = grad_expert_out;
  p.scale = recv_topk_weights;
  p.aux = expert_out;
  p.w_out = g_recv_topk_weights;
  cudaError_t e = ep::launch_combine_bwd_scaled(p, static_cast<int>(L->lay.pad_cap), sms,
                                                static_cast<cudaStream_t>(stream));
  g_launches.fetch_add(1, std::memory_order_relaxed);
  if (e != cudaSuccess) return cuda_fail(e, "ep_combine_weighted_bwd launch");
  return EP_OK;
}

ep_status_t ep_expert_offsets(ep_handle_t h, int32_t* offsets, void* stream) {
  const LayerInfo* L = nullptr;
  ep_status_t st = lookup(h, &L, 2);
  if (st != EP_OK) return st;
  if (L->rank_major)
    return fail(EP_ERR_INVALID_ARG, "layer %llu is rank-major: its expert offsets are the owner's single-buffer layer's",
                (unsigned long long)h.id);
  if (offsets == nullptr) return fail(EP_ERR_INVALID_ARG, "offsets is NULL");
  const int64_t own = L->nranks > 0 ? L->cfg.num_experts / L->nranks : L->cfg.num_experts;
  cudaError_t e = cudaMemcpyAsync(offsets, at<int>(h.mem, L->lay.offsets),
                                  static_cast<size_t>(own + 1) * 4,
                                  cudaMemcpyDeviceToDevice, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "ep_expert_offsets copy");
  return EP_OK;
}

ep_status_t ep_token_slots(ep_handle_t h, int32_t* slots, int64_t T, void* stream) {
  const LayerInfo* L = nullptr;
  ep_status_t st = lookup(h, &L, 2);
  if (st != EP_OK) return st;
  if ((st = check_tokens(L, T)) != EP_OK) return st;
  if (T == 0) return EP_OK;
  if (slots == nullptr) return fail(EP_ERR_INVALID_ARG, "slots is NULL");
  cudaError_t e = cudaMemcpyAsync(slots, at<int>(h.mem, L->lay.slot),
                                  static_cast<size_t>(T * L->cfg.top_k) * 4,
                                  cudaMemcpyDeviceToDevice, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "ep_token_slots copy");
  return EP_OK;
}

ep_status_t ep_read_info(ep_handle_t h, ep_info_t* info, void* stream) {
  const LayerInfo* L = nullptr;
  ep_status_t st = lookup(h, &L, 2);
  if (st != EP_OK) return st;
  if (info == nullptr) return fail(EP_ERR_INVALID_ARG, "info is NULL");
  int words[7] = {0, 0, 0, 0, 0, 0, 0};
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(words, h.mem, sizeof words, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "ep_read_info");
  if (words[ep::kHdrMagic] != ep::kPreparedMagic) {
    info->status = EP_ST_NOT_PREPARED | (words[ep::kHdrMagic] == ep::kTimedOutMagic ? EP_ST_TIMEOUT : 0u);
    info->num_tokens = info->used_rows = info->padding_rows = 0;
    return EP_OK;
  }
  info->status = static_cast<uint32_t>(words[ep::kHdrStatus]);
  info->num_tokens = words[ep::kHdrT];
  info->used_rows = words[ep::kHdrP];
  info->padding_rows = words[ep::kHdrNPad];
  return EP_OK;
}

ep_status_t ep_shard_count(ep_handle_t h, const int64_t* topk_idx, int64_t T, int32_t* local_counts,
                           void* stream) {
  const LayerInfo* L = nullptr;
  ep_status_t st = lookup(h, &L, 1);
  if (st != EP_OK) return st;
  if ((st = check_tokens(L, T)) != EP_OK) return st;
  if (T > 0 && topk_idx == nullptr) return fail(EP_ERR_INVALID_ARG, "topk_idx is NULL");
  if (topk_idx != nullptr && misaligned(topk_idx, 8)) return fail(EP_ERR_INVALID_ARG, "topk_idx is not 8-byte aligned");
  if (local_counts == nullptr) return fail(EP_ERR_INVALID_ARG, "local_counts is NULL");
  if (misaligned(local_counts, 4)) return fail(EP_ERR_INVALID_ARG, "local_counts is not 4-byte aligned");
  int sms = 0, mcs = 0;
  if ((st = check_device(&sms, nullptr, &mcs)) != EP_OK) return st;
  if ((st = check_shard_routes(L, T, mcs)) != EP_OK) return st;
  ep::RouteParams p = route_params(L, h, topk_idx, T, local_counts, 1);
  int launched = 0;
  cudaError_t e = ep::launch_shard_count(p, mcs, static_cast<cudaStream_t>(stream), &launched);
  g_launches.fetch_add(launched, std::memory_order_relaxed);
  if (e != cudaSuccess) return cuda_fail(e, "ep_shard_count launch");
  return EP_OK;
}

ep_status_t ep_shard_prepare(ep_handle_t h, const int64_t* topk_idx, int64_t T,
                             const int32_t* all_counts, int32_t* token_counts, int64_t alignment,
                             void* stream) {
  const LayerInfo* L = nullptr;
  ep_status_t st = lookup(h, &L, 1);
  if (st != EP_OK) return st;
  if ((st = check_tokens(L, T)) != EP_OK) return st;
  if (T > 0 && topk_idx == nullptr) return fail(EP_ERR_INVALID_ARG, "topk_idx is NULL");
  if (topk_idx != nullptr && misaligned(topk_idx, 8)) return fail(EP_ERR_INVALID_ARG, "topk_idx is not 8-byte aligned");
  if (all_counts == nullptr) return fail(EP_ERR_INVALID_ARG, "all_counts is NULL");
  if (misaligned(all_counts, 4)) return fail(EP_ERR_INVALID_ARG, "all_counts is not 4-byte aligned");
  if (token_counts == nullptr) return fail(EP_ERR_INVALID_ARG, "token_counts is NULL");
  if (misaligned(token_counts, 4)) return fail(EP_ERR_INVALID_ARG, "token_counts is not 4-byte aligned");
  if (alignment < 1 || alignment > L->cfg.max_alignment)
    return fail(EP_ERR_SHAPE, "alignment %lld outside [1, max_alignment=%lld]", (long long)alignment, (long long)L->cfg.max_alignment);
  int sms = 0, mcs = 0;
  if ((st = check_device(&sms, nullptr, &mcs)) != EP_OK) return st;
  if ((st = check_shard_routes(L, T, mcs)) != EP_OK) return st;
  ep::RouteParams p = route_params(L, h, topk_idx, T, token_counts, alignment);
  p.all_counts = all_counts;
  int launched = 0;
  cudaError_t e = ep::launch_shard_prepare(p, mcs, static_cast<cudaStream_t>(stream), &launched);
  g_launches.fetch_add(launched, std::memory_order_relaxed);
  if (e != cudaSuccess) return cuda_fail(e, "ep_shard_prepare launch");
  return EP_OK;
}

ep_status_t ep_shard_dispatch(ep_handle_t h, int64_t T, const void* tokens,
                              const float* topk_weights, void* const* recv_tokens,
                              float* const* recv_topk_weights, void* stream) {
  const LayerInfo* L = nullptr;
  ep_status_t st = lookup(h, &L, 1);
  if (st != EP_OK) return st;
  if ((st = check_tokens(L, T)) != EP_OK) return st;
  if ((st = check_payload(tokens, T, "tokens", T > 0)) != EP_OK) return st;
  if ((st = check_f32(topk_weights, "topk_weights", T > 0)) != EP_OK) return st;
  if ((st = check_table(recv_tokens, "recv_tokens")) != EP_OK) return st;
  if ((st = check_table(recv_topk_weights, "recv_topk_weights")) != EP_OK) return st;
  int sms = 0;
  if ((st = check_device(&sms)) != EP_OK) return st;
  ep::RowParams p = row_params(L, h, T);
  p.src = tokens;
  p.w_in = topk_weights;
  p.dst_tab = recv_tokens;
  p.wout_tab = recv_topk_weights;
  cudaError_t e = ep::launch_scatter_sharded(p, true, static_cast<int>(L->lay.pad_cap), sms,
                                             static_cast<cudaStream_t>(stream));
  g_launches.fetch_add(1, std::memory_order_relaxed);
  if (e != cudaSuccess) return cuda_fail(e, "ep_shard_dispatch launch");
  return EP_OK;
}

ep_status_t ep_shard_combine(ep_handle_t h, const void* const* expert_out, int64_t T, void* result,
                             void* stream) {
  const LayerInfo* L = nullptr;
  ep_status_t st = lookup(h, &L, 1);
  if (st != EP_OK) return st;
  if ((st = check_tokens(L, T)) != EP_OK) return st;
  if ((st = check_table(expert_out, "expert_out")) != EP_OK) return st;
  if ((st = check_payload(result, T, "result", T > 0)) != EP_OK) return st;
  int sms = 0;
  if ((st = check_device(&sms)) != EP_OK) return st;
  ep::RowParams p = row_params(L, h, T);
  p.src_tab = expert_out;
  p.dst = result;
  cudaError_t e = ep::launch_gather_sharded(p, false, sms, static_cast<cudaStream_t>(stream));
  g_launches.fetch_add(1, std::memory_order_relaxed);
  if (e != cudaSuccess) return cuda_fail(e, "ep_shard_combine launch");
  return EP_OK;
}

ep_status_t ep_shard_combine_bwd(ep_handle_t h, const void* grad, int64_t T,
                                 void* const* grad_expert_out, void* stream) {
  const LayerInfo* L = nullptr;
  ep_status_t st = lookup(h, &L, 1);
  if (st != EP_OK) return st;
  if ((st = check_tokens(L, T)) != EP_OK) return st;
  if ((st = check_payload(grad, T, "grad", T > 0)) != EP_OK) return st;
  if ((st = check_table(grad_expert_out, "grad_expert_out")) != EP_OK) return st;
  int sms = 0;
  if ((st = check_device(&sms)) != EP_OK) return st;
  ep::RowParams p = row_params(L, h, T);
  p.src = grad;
  p.dst_tab = grad_expert_out;
  cudaError_t e = ep::launch_scatter_sharded(p, false, static_cast<int>(L->lay.pad_cap), sms,
                                             static_cast<cudaStream_t>(stream));
  g_launches.fetch_add(1, std::memory_order_relaxed);
  if (e != cudaSuccess) return cuda_fail(e, "ep_shard_combine_bwd launch");
  return EP_OK;
}

ep_status_t ep_shard_dispatch_bwd(ep_handle_t h, const void* const* grad,
                                  const float* const* g_recv_topk_weights, int64_t T,
                                  void* grad_tokens, float* grad_topk_weights, void* stream) {
  const LayerInfo* L = nullptr;
  ep_status_t st = lookup(h, &L, 1);
  if (st != EP_OK) return st;
  if ((st = check_tokens(L, T)) != EP_OK) return st;
  if ((st = check_table(grad, "grad")) != EP_OK) return st;
  if (g_recv_topk_weights != nullptr && misaligned(g_recv_topk_weights, 8))
    return fail(EP_ERR_INVALID_ARG, "g_recv_topk_weights (table of per-rank addresses) is not 8-byte aligned");
  if ((st = check_payload(grad_tokens, T, "grad_tokens", T > 0)) != EP_OK) return st;
  if ((st = check_f32(grad_topk_weights, "grad_topk_weights", T > 0)) != EP_OK) return st;
  int sms = 0;
  if ((st = check_device(&sms)) != EP_OK) return st;
  ep::RowParams p = row_params(L, h, T);
  p.src_tab = grad;
  p.win_tab = g_recv_topk_weights;
  p.dst = grad_tokens;
  p.w_out = grad_topk_weights;
  cudaError_t e = ep::launch_gather_sharded(p, true, sms, static_cast<cudaStream_t>(stream));
  g_launches.fetch_add(1, std::memory_order_relaxed);
  if (e != cudaSuccess) return cuda_fail(e, "ep_shard_dispatch_bwd launch");
  return EP_OK;
}

ep_status_t ep_shard_token_owners(ep_handle_t h, int32_t* owners, int64_t T, void* stream) {
  const LayerInfo* L = nullptr;
  ep_status_t st = lookup(h, &L, 1);
  if (st != EP_OK) return st;
  if ((st = check_tokens(L, T)) != EP_OK) return st;
  if (T == 0) return EP_OK;
  if (owners == nullptr) return fail(EP_ERR_INVALID_ARG, "owners is NULL");
  cudaError_t e = cudaMemcpyAsync(owners, at<int>(h.mem, L->lay.dest),
                                  static_cast<size_t>(T * L->cfg.top_k) * 4,
                                  cudaMemcpyDeviceToDevice, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "ep_shard_token_owners copy");
  return EP_OK;
}

ep_status_t ep_register_layer_rank_major(ep_layer_config_t c, int64_t num_ranks, int64_t rank,
                                         uint64_t* id, size_t* handle_mem_size) {
  return register_rank_major(c, num_ranks, rank, id, handle_mem_size);
}

namespace {

// Shared checks of ep_rank_major_count / _prepare; launches the owners kernel.
ep_status_t rank_major_owners(const LayerInfo* L, const ep_handle_t& h, const int64_t* topk_idx, int64_t T,
                              ep::RouteParams* p, int* mcs, cudaStream_t s, int32_t* counts_user) {
  ep_status_t st = check_tokens(L, T);
  if (st != EP_OK) return st;
  if (T > 0 && topk_idx == nullptr) return fail(EP_ERR_INVALID_ARG, "topk_idx is NULL");
  if (topk_idx != nullptr && misaligned(topk_idx, 8)) return fail(EP_ERR_INVALID_ARG, "topk_idx is not 8-byte aligned");
  int sms = 0;
  if ((st = check_device(&sms, nullptr, mcs)) != EP_OK) return st;
  const long long lim = ep::shard_max_routes(static_cast<int>(L->nranks), *mcs);
  if (T * L->cfg.top_k > lim)
    return fail(EP_ERR_LIMIT, "%lld routes exceed the %lld a rank-major layer's routing map takes at %lld ranks on this device",
                (long long)(T * L->cfg.top_k), lim, (long long)L->nranks);
  *p = rank_major_route_params(L, h, topk_idx, T, counts_user);
  cudaError_t e = ep::launch_rank_major_owners(*p, sms, s);
  g_launches.fetch_add(1, std::memory_order_relaxed);
  if (e != cudaSuccess) return cuda_fail(e, "rank-major owners launch");
  return EP_OK;
}

}  // namespace

ep_status_t ep_rank_major_count(ep_handle_t h, const int64_t* topk_idx, int64_t T, int32_t* local_counts,
                                void* stream) {
  const LayerInfo* L = nullptr;
  ep_status_t st = lookup(h, &L, 3);
  if (st != EP_OK) return st;
  if (local_counts == nullptr) return fail(EP_ERR_INVALID_ARG, "local_counts is NULL");
  if (misaligned(local_counts, 4)) return fail(EP_ERR_INVALID_ARG, "local_counts is not 4-byte aligned");
  ep::RouteParams p;
  int mcs = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if ((st = rank_major_owners(L, h, topk_idx, T, &p, &mcs, s, local_counts)) != EP_OK) return st;
  int launched = 0;
  cudaError_t e = ep::launch_shard_count(p, mcs, s, &launched);
  g_launches.fetch_add(launched, std::memory_order_relaxed);
  if (e != cudaSuccess) return cuda_fail(e, "ep_rank_major_count launch");
  return EP_OK;
}

ep_status_t ep_rank_major_prepare(ep_handle_t h, const int64_t* topk_idx, int64_t T,
                                  const int32_t* all_counts, int32_t* recv_rows, void* stream) {
  const LayerInfo* L = nullptr;
  ep_status_t st = lookup(h, &L, 3);
  if (st != EP_OK) return st;
  if (all_counts == nullptr) return fail(EP_ERR_INVALID_ARG, "all_counts is NULL");
  if (misaligned(all_counts, 4)) return fail(EP_ERR_INVALID_ARG, "all_counts is not 4-byte aligned");
  if (recv_rows == nullptr) return fail(EP_ERR_INVALID_ARG, "recv_rows is NULL");
  if (misaligned(recv_rows, 4)) return fail(EP_ERR_INVALID_ARG, "recv_rows is not 4-byte aligned");
  ep::RouteParams p;
  int mcs = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if ((st = rank_major_owners(L, h, topk_idx, T, &p, &mcs, s, recv_rows)) != EP_OK) return st;
  p.all_counts = all_counts;
  int launched = 0;
  cudaError_t e = ep::launch_shard_prepare(p, mcs, s, &launched);
  g_launches.fetch_add(launched, std::memory_order_relaxed);
  if (e != cudaSuccess) return cuda_fail(e, "ep_rank_major_prepare launch");
  return EP_OK;
}

ep_status_t ep_rank_major_dispatch(ep_handle_t h, const int64_t* topk_idx, int64_t T, const void* tokens,
                                   const float* topk_weights, void* const* recv_tokens,
                                   int64_t* const* recv_topk_idx, float* const* recv_topk_weights,
                                   void* stream) {
  const LayerInfo* L = nullptr;
  ep_status_t st = lookup(h, &L, 3);
  if (st != EP_OK) return st;
  if ((st = check_tokens(L, T)) != EP_OK) return st;
  if (T > 0 && topk_idx == nullptr) return fail(EP_ERR_INVALID_ARG, "topk_idx is NULL");
  if (topk_idx != nullptr && misaligned(topk_idx, 8)) return fail(EP_ERR_INVALID_ARG, "topk_idx is not 8-byte aligned");
  if ((st = check_payload(tokens, T, "tokens", T > 0)) != EP_OK) return st;
  if (recv_topk_weights != nullptr && (st = check_f32(topk_weights, "topk_weights", T > 0)) != EP_OK) return st;
  if ((st = check_table(recv_tokens, "recv_tokens")) != EP_OK) return st;
  if ((st = check_table(recv_topk_idx, "recv_topk_idx")) != EP_OK) return st;
  if (recv_topk_weights != nullptr && (st = check_table(recv_topk_weights, "recv_topk_weights")) != EP_OK) return st;
  int sms = 0;
  if ((st = check_device(&sms)) != EP_OK) return st;
  ep::RowParams p = rank_major_row_params(L, h, T);
  p.src = tokens;
  p.dst_tab = recv_tokens;
  p.idx = reinterpret_cast<const long long*>(topk_idx);
  p.w_in = recv_topk_weights != nullptr ? topk_weights : nullptr;
  p.idx_tab = reinterpret_cast<long long* const*>(recv_topk_idx);
  p.wout_tab = recv_topk_weights;
  cudaError_t e = ep::launch_scatter_rank_major(p, sms, static_cast<cudaStream_t>(stream));
  g_launches.fetch_add(1, std::memory_order_relaxed);
  if (e != cudaSuccess) return cuda_fail(e, "ep_rank_major_dispatch launch");
  return EP_OK;
}

ep_status_t ep_rank_major_combine(ep_handle_t h, const void* const* partial, int64_t T, void* result,
                                  void* stream) {
  const LayerInfo* L = nullptr;
  ep_status_t st = lookup(h, &L, 3);
  if (st != EP_OK) return st;
  if ((st = check_tokens(L, T)) != EP_OK) return st;
  if ((st = check_table(partial, "partial")) != EP_OK) return st;
  if ((st = check_payload(result, T, "result", T > 0)) != EP_OK) return st;
  int sms = 0;
  if ((st = check_device(&sms)) != EP_OK) return st;
  ep::RowParams p = rank_major_row_params(L, h, T);
  p.src_tab = partial;
  p.dst = result;
  cudaError_t e = ep::launch_gather_sharded(p, false, sms, static_cast<cudaStream_t>(stream));
  g_launches.fetch_add(1, std::memory_order_relaxed);
  if (e != cudaSuccess) return cuda_fail(e, "ep_rank_major_combine launch");
  return EP_OK;
}

ep_status_t ep_rank_major_combine_bwd(ep_handle_t h, const void* grad, int64_t T, void* const* grad_recv,
                                      void* stream) {
  const LayerInfo* L = nullptr;
  ep_status_t st = lookup(h, &L, 3);
  if (st != EP_OK) return st;
  if ((st = check_tokens(L, T)) != EP_OK) return st;
  if ((st = check_payload(grad, T, "grad", T > 0)) != EP_OK) return st;
  if ((st = check_table(grad_recv, "grad_recv")) != EP_OK) return st;
  int sms = 0;
  if ((st = check_device(&sms)) != EP_OK) return st;
  ep::RowParams p = rank_major_row_params(L, h, T);
  p.src = grad;
  p.dst_tab = grad_recv;
  cudaError_t e = ep::launch_scatter_sharded(p, false, 0, sms, static_cast<cudaStream_t>(stream));
  g_launches.fetch_add(1, std::memory_order_relaxed);
  if (e != cudaSuccess) return cuda_fail(e, "ep_rank_major_combine_bwd launch");
  return EP_OK;
}

ep_status_t ep_rank_major_dispatch_bwd(ep_handle_t h, const void* const* grad_recv,
                                       const float* const* g_recv_topk_weights, int64_t T,
                                       void* grad_tokens, float* grad_topk_weights, void* stream) {
  const LayerInfo* L = nullptr;
  ep_status_t st = lookup(h, &L, 3);
  if (st != EP_OK) return st;
  if ((st = check_tokens(L, T)) != EP_OK) return st;
  if ((st = check_table(grad_recv, "grad_recv")) != EP_OK) return st;
  if (g_recv_topk_weights != nullptr && misaligned(g_recv_topk_weights, 8))
    return fail(EP_ERR_INVALID_ARG, "g_recv_topk_weights (table of per-rank addresses) is not 8-byte aligned");
  if ((st = check_payload(grad_tokens, T, "grad_tokens", T > 0)) != EP_OK) return st;
  if ((st = check_f32(grad_topk_weights, "grad_topk_weights", T > 0)) != EP_OK) return st;
  int sms = 0;
  if ((st = check_device(&sms)) != EP_OK) return st;
  ep::RowParams p = rank_major_row_params(L, h, T);
  p.src_tab = grad_recv;
  p.dst = grad_tokens;
  p.win_tab = g_recv_topk_weights;
  p.w_out = grad_topk_weights;
  cudaError_t e = ep::launch_gather_rank_major_bwd(p, sms, static_cast<cudaStream_t>(stream));
  g_launches.fetch_add(1, std::memory_order_relaxed);
  if (e != cudaSuccess) return cuda_fail(e, "ep_rank_major_dispatch_bwd launch");
  return EP_OK;
}

}  // extern "C"
