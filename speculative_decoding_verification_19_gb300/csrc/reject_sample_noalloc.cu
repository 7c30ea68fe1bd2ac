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
#include <string.h>

#include <atomic>

#include "common.cuh"
#include "reject_sample.cuh"

namespace specv {

// Scratch of the no-allocation path: a 256-byte status area, the chunk
// statistics, the per-request draw states and the residual chunk masses.
// Every GPU that loads the library holds it until exit.
constexpr size_t kNoAllocScratchBytes = (size_t)1 << 20;  // 1 MiB
constexpr size_t kNoAllocStatusBytes = 256;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 256;
static std::atomic<void*> g_noalloc_ptr[kMaxDevices];

// Device address of the scratch array on the current device, looked up once
// per device (the host-side symbol is not a device address).
static spec_status noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SPEC_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return SPEC_ERR_UNSUPPORTED;
  void* p = g_noalloc_ptr[dev].load(std::memory_order_acquire);
  if (p == nullptr) {
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return SPEC_ERR_CUDA;
    g_noalloc_ptr[dev].store(p, std::memory_order_release);
  }
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
  if (dims == nullptr || dims->B < 1 || dims->M < 1 || dims->V < 1) return SPEC_ERR_INVALID_ARG;
  if (dims->M > 64 || dims->V > rs_max_vocab(dims->logits_dtype)) return SPEC_ERR_UNSUPPORTED;
  if (dims->logits_dtype != SPEC_BF16 && dims->logits_dtype != SPEC_F32) return SPEC_ERR_INVALID_ARG;
  if (!target_logits || !draft_logits || !tokens || !temperature || !out_tokens || !path ||
      !accepted_len)
    return SPEC_ERR_INVALID_ARG;
  // the statistics of every (request, row, chunk) must fit the fixed scratch
  WsLayout lay;
  memset(&lay, 0, sizeof(lay));
  lay.status_off = 0;
  lay.rs_off = kNoAllocStatusBytes;
  lay.rs_chunk = rs_chunk_elems(dims->logits_dtype);
  lay.rs_chunks = (int)ceil_div64(dims->V, lay.rs_chunk);
  lay.rs_bytes = sizeof(RowStat) * (size_t)dims->B * 2 * dims->M * lay.rs_chunks;
  lay.rs_draw_off = (lay.rs_off + lay.rs_bytes + 255) / 256 * 256;
  lay.rs_zsum_off = (lay.rs_draw_off + sizeof(DrawState) * (size_t)dims->B + 255) / 256 * 256;
  lay.total = lay.rs_zsum_off + sizeof(double) * (size_t)dims->B * lay.rs_chunks;
  if (lay.total > kNoAllocScratchBytes) return SPEC_ERR_UNSUPPORTED;

  void* scratch = nullptr;
  const spec_status s = noalloc_scratch(&scratch);
  if (s != SPEC_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the status word starts each call at zero; the rest needs no clearing
  // (every entry read is written earlier in the same call)
  if (cudaMemsetAsync(scratch, 0, kNoAllocStatusBytes, st) != cudaSuccess) return SPEC_ERR_CUDA;

  RsArgs a;
  a.target = target_logits;
  a.draft = draft_logits;
  a.tokens = tokens;
  a.parent = parent;
  a.temperature = temperature;
  a.seed = seed;
  a.offset = offset;
  a.b_base = b_base;
  a.out_tokens = out_tokens;
  a.path = path;
  a.accepted_len = accepted_len;
  a.probe = probe;
  a.d = *dims;
  a.ws = scratch;
  int launches = 0;
  return rs_launch(a, lay, st, &launches) == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}
