// mla_decode_noalloc: mla_decode for callers that cannot allocate device
// memory.
//
// mla_decode needs a workspace for its split-KV partials, tile plan and error
// word, and normally the caller allocates it.  Some callers cannot: a plugin
// running inside a host application that owns the whole device memory pool
// and gives the plugin no allocator, or a serving loop that must never call
// cudaMalloc because the call can block and synchronise the device.  For
// them this entry point takes the workspace from one fixed array compiled
// into the library (g_noalloc_scratch below).  Every GPU that loads the
// library holds that array until the process exits.
//
// The array's name in host code is only a host-side stand-in for the symbol,
// never a device address.  The device address is looked up with
// cudaGetSymbolAddress, with the caller's device current, on every call: the
// lookup allocates nothing, and a fresh lookup stays right after the device
// or its primary context has been reset (which reloads the module and can
// move the array).  The first lookup on a device loads the library's module
// there, so that first call must not be made during stream capture.
#include "internal.cuh"

namespace mla {
namespace {

constexpr size_t kNoAllocBytes = MLA_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

// Device address of the scratch array on the current device.
mla_status scratch_for_current_device(void **out) {
  void *p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
    return MLA_ERR_CUDA;
  *out = p;
  return MLA_OK;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace
}  // namespace mla

extern "C" __attribute__((visibility("default"))) mla_status mla_decode_noalloc(
    const void *q_lat, const void *q_rope, const void *cache, int num_blocks,
    const int32_t *block_table, int max_blocks, const int32_t *seqlens, int max_seqlen, int B,
    int Hq, const mla_dims *dims, void *o_lat, float *lse, mla_stream_t stream) {
  using namespace mla;
  // 1. size check before anything touches the GPU
  size_t need = 0;
  const mla_status s = mla_decode_workspace_size(B, Hq, max_seqlen, dims, &need);
  if (s != MLA_OK) return s;
  if (need > kNoAllocBytes) return MLA_ERR_WORKSPACE;
  if (B == 0) return MLA_OK;
  // 2. the same argument checks as mla_decode, so that a bad call launches
  //    nothing (not even the header clear below)
  if (num_blocks < 1 || max_blocks < 1 || !q_lat || !cache || !block_table || !seqlens ||
      !o_lat || !lse || (dims->d_r > 0 && !q_rope))
    return MLA_ERR_INVALID_ARG;
  if (!aligned(q_lat, 16) || (q_rope && !aligned(q_rope, 16)) || !aligned(cache, 128) ||
      !aligned(o_lat, 16) || !aligned(lse, 4) || !aligned(block_table, 4) ||
      !aligned(seqlens, 4))
    return MLA_ERR_INVALID_ARG;
  // 3. the shared scratch keeps the previous call's contents: clear its
  //    header (the device error word) before this call's kernels run
  void *scratch = nullptr;
  const mla_status t = scratch_for_current_device(&scratch);
  if (t != MLA_OK) return t;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(scratch, 0, kWsHeader, st) != cudaSuccess) return MLA_ERR_CUDA;
  // 4. the regular decode, with the scratch array as its workspace
  return mla_decode(q_lat, q_rope, cache, num_blocks, block_table, max_blocks, seqlens,
                    max_seqlen, B, Hq, dims, o_lat, lse, scratch, kNoAllocBytes, stream);
}

extern "C" __attribute__((visibility("default"))) mla_status mla_decode_noalloc_get_error(
    mla_stream_t stream) {
  using namespace mla;
  void *scratch = nullptr;
  const mla_status t = scratch_for_current_device(&scratch);
  if (t != MLA_OK) return t;
  // the array's first 256 bytes are a decode workspace header like any other
  return mla_get_error(scratch, stream);
}
