// grpo_static.cu -- grpo_loss_fwd_bwd without a caller-provided workspace.
//
// Some callers cannot allocate device memory at the point where they need
// the loss: code that runs while a CUDA stream is being captured into a graph
// (cudaMalloc is not a capturable operation), hosts whose device memory is
// entirely owned by another allocator (a framework's caching pool, an
// inference server's fixed partitions), or latency-critical loops where a
// cudaMalloc / cudaFree pair (cudaFree synchronises the device) is not
// acceptable.  For them, grpo_loss_fwd_bwd_static runs the same fused
// forward + backward with its scratch memory taken from a fixed array that
// lives in this library's device image.
//
// The array is file-scope device memory of kStaticScratchBytes: every GPU
// that loads the library holds it until the process exits.  All calls share
// it and it keeps the last call's contents; the entry point clears what must
// start at zero (the header's status word and counters, through the same
// memset as the workspace path) and overwrites the rest before reading it.  Because the array is shared, calls whose work overlaps on the
// GPU (different streams, or different host threads, without ordering
// between them) race on it: serialise them.
#include <mutex>

#include "grpo_internal.cuh"

namespace {

constexpr size_t kStaticScratchBytes = (size_t)9 << 19;  // 4.5 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

// Per-device device address of g_static_scratch.  In host code the array's
// name is only a stand-in; the address a kernel may use comes from
// cudaGetSymbolAddress, taken with that device current.  The address belongs
// to the device's context: after cudaDeviceReset the runtime makes a new
// primary context, where the array may sit elsewhere.  So each cached address
// is stored with the unique id of the context it was taken in (cuCtxGetId,
// reached through the runtime's driver entry-point query, so the library does
// not link the driver library itself), and looked up again when the current
// context's id differs.
std::mutex g_setup_mutex;
struct Cached {
  unsigned long long ctx_id = 0;  // 0: nothing cached
  void* addr = nullptr;
};
Cached g_scratch[kMaxDevices];

typedef int (*CtxGetCurrentFn)(void** ctx);                      // cuCtxGetCurrent
typedef int (*CtxGetIdFn)(void* ctx, unsigned long long* id);    // cuCtxGetId
CtxGetCurrentFn g_ctx_current = nullptr;
CtxGetIdFn g_ctx_id = nullptr;

// The current context's unique id, or 0 when it cannot be read (no current
// context yet, or a driver without the queries).
unsigned long long current_ctx_id() {
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      g_ctx_current = (CtxGetCurrentFn)f;
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      g_ctx_id = (CtxGetIdFn)f;
  });
  if (!g_ctx_current || !g_ctx_id) return 0;
  void* ctx = nullptr;
  unsigned long long id = 0;
  if (g_ctx_current(&ctx) != 0 || ctx == nullptr) return 0;
  if (g_ctx_id(ctx, &id) != 0) return 0;
  return id;
}

grpo_status_t scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GRPO_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  Cached& c = g_scratch[dev];
  const unsigned long long id = current_ctx_id();
  if (c.addr == nullptr || id == 0 || id != c.ctx_id) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr)
      return GRPO_ERR_CUDA;
    c.addr = p;
    // the lookup above makes the device's primary context current if it was not
    c.ctx_id = id != 0 ? id : current_ctx_id();
  }
  *out = c.addr;
  return GRPO_OK;
}

}  // namespace

extern "C" grpo_status_t grpo_loss_fwd_bwd_static(
    const void* policy_logits, const void* ref_logits, grpo_dtype_t dt, int64_t B, int64_t T,
    int64_t V, const int64_t* action_ids, const float* old_logps,
    const uint8_t* completion_mask, const float* rewards, const grpo_groups_t* groups,
    const grpo_params_t* params, void* grad_logits, float* out3, float* per_seq,
    float* logps_out, float* adv_out, void* stream) {
  // sizes beyond the fixed scratch are rejected before anything else runs;
  // a shard call lays its scratch out for the whole batch (groups->num_seqs)
  if (B < 0 || T < 0 || T > ((int64_t)1 << 30)) return GRPO_ERR_SHAPE;
  const int64_t Bw = (params && params->shard && groups && groups->num_seqs > B) ? groups->num_seqs : B;
  if (grpo_workspace_size(Bw, T, 0) > kStaticScratchBytes) return GRPO_ERR_WORKSPACE;
  void* ws = nullptr;
  const grpo_status_t st = scratch_for_current_device(&ws);
  if (st != GRPO_OK) return st;
  return grpo_loss_fwd_bwd(policy_logits, ref_logits, dt, B, T, V, action_ids, old_logps,
                           completion_mask, rewards, groups, params, grad_logits, out3, per_seq,
                           logps_out, adv_out, ws, kStaticScratchBytes, stream);
}
