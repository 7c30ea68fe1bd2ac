// KV commit: roll the cache back to the accepted prefix, or compact the
// accepted path of a draft tree (page 2 §3.3 rollback after a partial
// acceptance; page 2 §5.4 and page 3 tree section: the dynamic rollback path).
//
// One CTA per request; each thread owns fixed 16-byte lanes of fixed KV
// heads and walks j = 1..a in increasing order, moving slot ctx+path[j] to
// slot ctx+j.  In-place is safe: path[j] >= j, so slot ctx+j is written at
// step j only after every source that could equal it (path[k] = j needs
// k < j) has been read by the same thread at an earlier step.  A chain
// (path[j] = j) moves nothing.
#include "common.cuh"
#include "kv_commit.cuh"

namespace specv {

template <typename T>
__global__ void __launch_bounds__(256) kv_commit_kernel(
    T* k_cache, T* v_cache, const int32_t* __restrict__ block_table, const int32_t* ctx_lens,
    int32_t* new_ctx_lens, const int32_t* path, const int32_t* accepted_len, spec_dims d,
    uint32_t* __restrict__ status) {
  pdl_trigger();
  pdl_wait();  // path and accepted_len come from the previous kernel
  const int b = blockIdx.x, tid = threadIdx.x;
  const int ctx = ctx_lens[b];
  const int a = accepted_len[b];
  const int32_t* pth = path + (int64_t)b * d.M;
  const int32_t* bt = block_table + (int64_t)b * d.max_blocks;

  const bool bad_cap = a >= 0 && (ctx < 0 || (int64_t)ctx + d.M > (int64_t)d.max_blocks * kBlock);
  int bad_path = a >= d.M;
  int bad_block = 0;
  if (a >= 0 && !bad_cap && !bad_path) {
    for (int j = tid; j <= a; j += blockDim.x) {
      const int pj = pth[j];
      bad_path |= (j == 0) ? (pj != 0) : (pj < j || pj >= d.M);
    }
    const int p0 = ctx / kBlock, p1 = (ctx + d.M - 1) / kBlock;
    for (int p = p0 + tid; p <= p1; p += blockDim.x) {
      const int id = bt[p];
      bad_block |= (id < 0 || id >= d.num_blocks);
    }
  }
  bad_path = __syncthreads_or(bad_path);
  bad_block = __syncthreads_or(bad_block);
  const bool bad = bad_cap || bad_path || bad_block;
  if (a >= 0 && !bad) {
    constexpr int kVec = 16 / sizeof(T);
    const int lanes = d.D / kVec;
    const int work = d.Hkv * lanes;
    for (int w = tid; w < work; w += blockDim.x) {
      const int lane = w % lanes, h = w / lanes;
      for (int j = 1; j <= a; ++j) {
        const int src = ctx + pth[j], dst = ctx + j;
        if (src == dst) continue;
        const int64_t so = (((int64_t)bt[src / kBlock] * d.Hkv + h) * kBlock + src % kBlock) * d.D;
        const int64_t dof = (((int64_t)bt[dst / kBlock] * d.Hkv + h) * kBlock + dst % kBlock) * d.D;
        const uint4 kv = reinterpret_cast<const uint4*>(k_cache + so)[lane];
        const uint4 vv = reinterpret_cast<const uint4*>(v_cache + so)[lane];
        reinterpret_cast<uint4*>(k_cache + dof)[lane] = kv;
        reinterpret_cast<uint4*>(v_cache + dof)[lane] = vv;
      }
    }
  }
  __syncthreads();  // every thread has read ctx_lens[b] (new_ctx_lens may alias it)
  if (tid == 0) {
    if (bad_cap) raise_status(status, SPEC_ERR_CAPACITY);
    if (bad_path) raise_status(status, SPEC_ERR_INVALID_ARG);
    if (bad_block) raise_status(status, SPEC_ERR_DEVICE_BOUNDS);
    new_ctx_lens[b] = (a >= 0 && !bad) ? ctx + a + 1 : ctx;
  }
}

template <typename T>
static cudaError_t launch_commit_t(const CommitArgs& a, const WsLayout& lay, cudaStream_t st,
                                   int* launches) {
  uint32_t* status = reinterpret_cast<uint32_t*>(static_cast<char*>(a.ws) + lay.status_off);
  PdlLaunch L(dim3(a.d.B), dim3(256), 0, st);
  const cudaError_t e = cudaLaunchKernelEx(&L.cfg, kv_commit_kernel<T>, static_cast<T*>(a.k_cache),
                                           static_cast<T*>(a.v_cache), a.block_table, a.ctx_lens,
                                           a.new_ctx_lens, a.path, a.accepted_len, a.d, status);
  ++*launches;
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t commit_launch(const CommitArgs& a, const WsLayout& lay, cudaStream_t st, int* launches) {
  if (a.d.kv_dtype == SPEC_BF16) return launch_commit_t<__nv_bfloat16>(a, lay, st, launches);
  return launch_commit_t<float>(a, lay, st, launches);
}

}  // namespace specv
