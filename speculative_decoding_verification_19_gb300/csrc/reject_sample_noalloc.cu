// spec_reject_sample_noalloc: the accept / reject / resample step for callers
// that cannot hand the library a device workspace.
//
// Some callers cannot allocate device memory on the call path: cudaMalloc
// may synchronise the whole device, is not allowed while a stream is being
// captured, and serving engines that carve all of HBM into a fixed KV-cache
// pool at start-up often have no allocator left to call.  This entry point
// therefore keeps its scratch (the per-chunk row statistics and the status
// word) in a fixed-size array in the library's own device memory instead of
// a caller-provided workspace, and runs the same kernels as
// spec_reject_sample.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <string.h>

#include <mutex>

#include "common.cuh"
#include "reject_sample.cuh"

namespace specv {

// Scratch of the no-allocation path: a 256-byte status area, the chunk
// statistics, the per-request draw states and the residual chunk masses.
// Every GPU that loads the library holds it until exit.
constexpr size_t kNoAllocScratchBytes = (size_t)1 << 20;  // 1 MiB
constexpr size_t kNoAllocStatusBytes = 256;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the scratch array in the current CUDA context.  The
// host-side symbol is not a device address, and the array's address belongs
// to the context that loaded the module: after cudaDeviceReset, or under
// another context on the same device, the module is loaded again elsewhere.
// So the address is cached per context, keyed by the context's unique id,
// and looked up (cudaGetSymbolAddress) the first time a context is seen.
struct CtxAddr {
  unsigned long long ctx_id;
  void* ptr;
};
constexpr int kMaxContexts = 64;
static std::mutex g_noalloc_mu;
static CtxAddr g_noalloc_cache[kMaxContexts];
static int g_noalloc_n = 0;

static PFN_cuCtxGetCurrent_v4000 ctx_current_fn() {
  static PFN_cuCtxGetCurrent_v4000 fn = nullptr;
  if (fn == nullptr) {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
  }
  return fn;
}
static PFN_cuCtxGetId_v12000 ctx_id_fn() {
  static PFN_cuCtxGetId_v12000 fn = nullptr;
  if (fn == nullptr) {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
  }
  return fn;
}

static spec_status noalloc_scratch(void** out) {
  auto get_ctx = ctx_current_fn();
  auto get_id = ctx_id_fn();
  if (get_ctx == nullptr || get_id == nullptr) return SPEC_ERR_CUDA;
  CUcontext ctx = nullptr;
  if (get_ctx(&ctx) != CUDA_SUCCESS) return SPEC_ERR_CUDA;
  if (ctx == nullptr) {
    // no context is current yet: the runtime makes the device's primary
    // context current on its first call that needs one, such as this lookup
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return SPEC_ERR_CUDA;
    if (get_ctx(&ctx) != CUDA_SUCCESS || ctx == nullptr) return SPEC_ERR_CUDA;
  }
  unsigned long long id = 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return SPEC_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  for (int i = 0; i < g_noalloc_n; ++i)
    if (g_noalloc_cache[i].ctx_id == id) {
      *out = g_noalloc_cache[i].ptr;
      return SPEC_OK;
    }
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
    return SPEC_ERR_CUDA;
  // a full table forgets its oldest entry (a context id is never reused)
  if (g_noalloc_n == kMaxContexts) {
    memmove(g_noalloc_cache, g_noalloc_cache + 1, sizeof(CtxAddr) * (kMaxContexts - 1));
    --g_noalloc_n;
  }
  g_noalloc_cache[g_noalloc_n++] = CtxAddr{id, p};
  *out = p;
  return SPEC_OK;
}

}  // namespace specv

using namespace specv;

extern "C" spec_status spec_reject_sample_noalloc(
    const void* target_logits, const void* draft_logits, const int32_t* tokens,
    const int32_t* parent, const float* temperature, uint64_t seed, uint64_t offset,
    uint64_t b_base, int32_t* out_tokens, int32_t* path, int32_t* accepted_len, float* probe,
    const spec_dims* dims, void* stream) {
  // the same dims checks as spec_reject_sample
  const spec_status chk = check_common(dims);
  if (chk != SPEC_OK) return chk;
  if (dims->V < 1) return SPEC_ERR_INVALID_ARG;
  if (dims->V > rs_max_vocab(dims->logits_dtype)) return SPEC_ERR_UNSUPPORTED;
  if (!target_logits || !draft_logits || !tokens || !temperature || !out_tokens || !path ||
      !accepted_len)
    return SPEC_ERR_INVALID_ARG;
  // The call runs the kernels spec_reject_sample would run on these inputs
  // and dims->reject_impl: the one-kernel path when asked for (and the
  // shape allows it), else the staged ones.  Each has its own scratch
  // layout, which must fit the fixed array.
  const int esz = dims->logits_dtype == SPEC_BF16 ? 2 : 4;
  const bool aligned = ((size_t)dims->V * esz) % 16 == 0 &&
                       (reinterpret_cast<uintptr_t>(target_logits) % 16) == 0 &&
                       (reinterpret_cast<uintptr_t>(draft_logits) % 16) == 0;
  const bool fused = dims->reject_impl == SPEC_REJECT_FUSED &&
                     rso_supported(*dims, aligned, parent == nullptr);
  if (dims->reject_impl == SPEC_REJECT_FUSED && !fused) return SPEC_ERR_UNSUPPORTED;
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  // status, the chunk statistics, the draw states, the residual chunk
  // masses, the chain tail's counters; for the one-kernel path also its
  // control words, row normalisers and counters
  WsLayout lay;
  memset(&lay, 0, sizeof(lay));
  lay.status_off = 0;
  lay.rs_chunk = rs_chunk_elems(dims->logits_dtype);
  lay.rs_chunks = (int)ceil_div64(dims->V, lay.rs_chunk);
  lay.rs_off = kNoAllocStatusBytes;
  lay.rs_bytes = sizeof(RowStat) * (size_t)dims->B * 2 * dims->M * lay.rs_chunks;
  lay.rs_draw_off = up(lay.rs_off + lay.rs_bytes);
  lay.rs_zsum_off = up(lay.rs_draw_off + sizeof(DrawState) * (size_t)dims->B);
  lay.rs_tail_off = up(lay.rs_zsum_off + sizeof(double) * (size_t)dims->B * lay.rs_chunks);
  lay.total = lay.rs_tail_off + sizeof(uint32_t) * (2 * (size_t)dims->B + 2);
  if (fused) lay.total = rsf_layout(*dims, up(lay.total), &lay);
  if (lay.total > kNoAllocScratchBytes) return SPEC_ERR_UNSUPPORTED;

  void* scratch = nullptr;
  const spec_status s = noalloc_scratch(&scratch);
  if (s != SPEC_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // The status word and the counters start each call at zero, whatever an
  // earlier call (one whose wait gave up, say) left there.  Everything else
  // read is written earlier in the same call.
  char* sb = static_cast<char*>(scratch);
  if (cudaMemsetAsync(sb, 0, kNoAllocStatusBytes, st) != cudaSuccess) return SPEC_ERR_CUDA;
  if (cudaMemsetAsync(sb + lay.rs_tail_off, 0, sizeof(uint32_t) * (2 * (size_t)dims->B + 2), st) !=
      cudaSuccess)
    return SPEC_ERR_CUDA;
  if (fused && cudaMemsetAsync(sb + lay.rsf_ctl_off, 0, lay.total - lay.rsf_ctl_off, st) !=
                   cudaSuccess)
    return SPEC_ERR_CUDA;

  RsArgs a;
  a.target = target_logits;
  a.draft = draft_logits;
  a.tokens = tokens;
  a.parent = parent;
  a.temperature = temperature;
  a.top_k = nullptr;
  a.top_p = nullptr;
  a.seed = seed;
  a.offset = offset;
  a.b_base = b_base;
  a.out_tokens = out_tokens;
  a.path = path;
  a.accepted_len = accepted_len;
  a.probe = probe;
  a.d = *dims;
  a.d.reject_impl = fused ? SPEC_REJECT_FUSED : SPEC_REJECT_STAGED;
  a.ws = scratch;
  int launches = 0;
  return rs_launch(a, lay, st, &launches) == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}
