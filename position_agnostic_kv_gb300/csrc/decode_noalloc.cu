// lazy_attn_decode_noalloc: the split-KV decode for callers that cannot allocate device memory.
//
// Some hosts own every byte of GPU memory themselves: an inference engine that reserves all
// of HBM for its KV pool when it starts and hands plugins no allocator, or a latency-bound
// decode loop that must never call cudaMalloc (which may synchronise the device and take
// milliseconds).  Such callers cannot provide the workspace that lazy_attn_decode needs for
// its per-split partial results.  This entry point keeps that workspace in a fixed array
// compiled into the library instead, so neither the caller nor the library allocates.
//
// The array is g_decode_scratch below: kNoAllocScratchBytes (16 MiB) per GPU, held by every
// GPU that loads the library until the process exits.  In host code its name only stands in
// for the symbol; the device address comes from cudaGetSymbolAddress, looked up once per
// device (the first call on each device does it, with that device current).
#include <mutex>

#include "decode.cuh"

namespace lazykv {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;

static __device__ __align__(256) uint8_t g_decode_scratch[kNoAllocScratchBytes];

namespace {
std::mutex g_scratch_mu;
constexpr int kMaxDev = 64;
void* g_scratch_addr[kMaxDev] = {};
}  // namespace

// Device address of g_decode_scratch on the current device (looked up on first use).
static int scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(LAZY_ECUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDev) return fail(LAZY_EINVAL, "device index %d too large", dev);
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess || p == nullptr)
      return fail(LAZY_ECUDA, "cudaGetSymbolAddress(decode scratch): %s", cudaGetErrorString(e));
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return LAZY_OK;
}

}  // namespace lazykv

using namespace lazykv;

extern "C" int lazy_attn_decode_noalloc(const void* q, const int32_t* seq_len, const int32_t* q_start,
                                        const int32_t* doc_blocks, const uint64_t* meta, int B,
                                        int max_blocks, const void* k_cache, const void* v_cache,
                                        int num_pages, int Hq, int Hkv, int D, float scale,
                                        const lazy_pos_cfg* cfg, void* out, float* lse, void* stream) {
  int rc = check_device();
  if (rc) return rc;
  if (B < 0 || max_blocks <= 0 || Hq <= 0 || Hkv <= 0 || (Hq % Hkv) != 0 || (D != 64 && D != 128))
    return fail(LAZY_EINVAL, "bad decode sizes (B=%d max_blocks=%d Hq=%d Hkv=%d D=%d)", B, max_blocks, Hq,
                Hkv, D);
  if (B == 0) return LAZY_OK;
  const size_t need = decode_ws_bytes(B, Hq, Hkv, D, max_blocks);
  if (need > kNoAllocScratchBytes)
    return fail(LAZY_EINVAL,
                "lazy_attn_decode_noalloc: this batch needs %zu bytes of split scratch but the fixed "
                "array holds %zu; use lazy_attn_decode with a caller workspace",
                need, kNoAllocScratchBytes);
  void* scratch = nullptr;
  if (need > 0) {
    rc = scratch_address(&scratch);
    if (rc) return rc;
  }
  // Nothing in the scratch has to start at zero: every partial (O, m, l) that the merge reads
  // is written earlier in the same call.
  return lazy_attn_decode(q, seq_len, q_start, doc_blocks, meta, B, max_blocks, k_cache, v_cache, num_pages, Hq,
                          Hkv, D, scale, cfg, out, lse, scratch, need > 0 ? kNoAllocScratchBytes : 0, stream);
}
