// Host helpers of liblazykv: error messages, the device status word, device checks and the
// preparation of positional parameters (RoPE / YaRN frequencies, softmax scale).
#include <cmath>
#include <cstdarg>
#include <cstring>
#include <mutex>

#include "common.cuh"

namespace lazykv {

// One status word per GPU that loads the library.  Kernels OR LAZY_STATUS_* bits into it;
// lazy_device_status reads and clears it.
__device__ uint32_t g_status_word;

static thread_local char t_msg[512] = "";

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_msg, sizeof(t_msg), fmt, ap);
  va_end(ap);
  return code;
}

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_mu;
uint32_t* g_status_ptr[kMaxDevices] = {};
int g_sms[kMaxDevices] = {};
int g_cc_major[kMaxDevices] = {};
}  // namespace

static int current_device(int* dev) {
  cudaError_t e = cudaGetDevice(dev);
  if (e != cudaSuccess) return fail(LAZY_ECUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (*dev < 0 || *dev >= kMaxDevices) return fail(LAZY_EINVAL, "device index %d too large", *dev);
  return LAZY_OK;
}

static int ensure_device_info(int dev) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_sms[dev] == 0) {
    cudaDeviceProp p;
    cudaError_t e = cudaGetDeviceProperties(&p, dev);
    if (e != cudaSuccess) return fail(LAZY_ECUDA, "cudaGetDeviceProperties: %s", cudaGetErrorString(e));
    g_sms[dev] = p.multiProcessorCount;
    g_cc_major[dev] = p.major;
  }
  if (g_status_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&ptr, g_status_word);
    if (e != cudaSuccess) return fail(LAZY_ECUDA, "cudaGetSymbolAddress(status): %s", cudaGetErrorString(e));
    g_status_ptr[dev] = static_cast<uint32_t*>(ptr);
  }
  return LAZY_OK;
}

int check_device() {
  int dev = 0;
  int rc = current_device(&dev);
  if (rc) return rc;
  rc = ensure_device_info(dev);
  if (rc) return rc;
  if (g_cc_major[dev] != 10)
    return fail(LAZY_EARCH, "liblazykv is built for sm_103a; current device is CC %d.x", g_cc_major[dev]);
  return LAZY_OK;
}

int sm_count() {
  int dev = 0;
  if (current_device(&dev) || ensure_device_info(dev)) return 148;
  return g_sms[dev];
}

uint32_t* status_word() {
  int dev = 0;
  if (current_device(&dev) || ensure_device_info(dev)) return nullptr;
  return g_status_ptr[dev];
}

int prepare_pos(const lazy_pos_cfg* cfg, int Hq, int D, float scale, PosParams* out) {
  if (!cfg) return fail(LAZY_EINVAL, "pos cfg is NULL");
  std::memset(out, 0, sizeof(*out));
  out->kind = cfg->kind;
  out->rotary_dim = cfg->rotary_dim;
  out->slopes = cfg->alibi_slopes;
  out->table = cfg->cos_sin;
  out->max_pos = cfg->cos_sin ? cfg->max_pos : 0;
  out->interleaved = cfg->interleaved != 0;
  if (cfg->kind < LAZY_POS_ROPE || cfg->kind > LAZY_POS_NONE)
    return fail(LAZY_EINVAL, "unknown positional kind %d", cfg->kind);
  const bool rotary = cfg->kind == LAZY_POS_ROPE || cfg->kind == LAZY_POS_YARN;
  double s = 1.0 / std::sqrt(double(D));
  if (rotary) {
    const int rd = cfg->rotary_dim;
    if (rd < 16 || rd > D || rd % 16)
      return fail(LAZY_EINVAL, "rotary_dim (%d) must be a multiple of 16 in [16, head_dim = %d]", rd, D);
    if (!(cfg->rope_theta > 1.0f)) return fail(LAZY_EINVAL, "rope_theta must be > 1");
    const int half = rd / 2;
    const double two_pi = 6.283185307179586476925286766559;
    double factor = cfg->yarn_factor, bf = cfg->yarn_beta_fast, bs = cfg->yarn_beta_slow;
    if (cfg->kind == LAZY_POS_YARN) {
      if (!(factor >= 1.0) || cfg->yarn_orig_ctx <= 0)
        return fail(LAZY_EINVAL, "YaRN needs yarn_factor >= 1 and yarn_orig_ctx > 0");
      if (bf == 0.0) bf = 32.0;
      if (bs == 0.0) bs = 1.0;
      if (!(bf > bs)) return fail(LAZY_EINVAL, "YaRN needs beta_fast > beta_slow");
    }
    for (int i = 0; i < half; ++i) {
      double theta = std::pow(double(cfg->rope_theta), -2.0 * i / double(rd));
      if (cfg->kind == LAZY_POS_YARN) {
        // NTK-by-parts ramp of the YaRN paper: gamma = clamp((L0/lambda - b_slow)/(b_fast - b_slow))
        const double ratio = double(cfg->yarn_orig_ctx) * theta / two_pi;  // L0 / lambda_i
        double gamma = (ratio - bs) / (bf - bs);
        gamma = gamma < 0.0 ? 0.0 : (gamma > 1.0 ? 1.0 : gamma);
        theta = (1.0 - gamma) * theta / factor + gamma * theta;
      }
      const double turns = theta / two_pi;  // < 1 / (2 pi) since theta <= 1
      out->turns[i] = (unsigned long long)std::ldexp(turns, 64);
    }
    if (cfg->kind == LAZY_POS_YARN && factor > 1.0) {
      const double mscale = 0.1 * std::log(factor) + 1.0;
      s *= mscale * mscale;
    }
  } else if (cfg->kind == LAZY_POS_ALIBI) {
    if (!cfg->alibi_slopes) return fail(LAZY_EINVAL, "ALiBi needs alibi_slopes");
  }
  if (scale != 0.0f) s = scale;
  out->scale_log2 = float(s * 1.4426950408889634073599246810019);
  (void)Hq;
  return LAZY_OK;
}

}  // namespace lazykv

extern "C" {

const char* lazy_last_error(void) { return lazykv::t_msg; }

int lazy_version(void) { return 100; }

int lazy_device_status(void* stream, uint32_t* status) {
  using namespace lazykv;
  if (!status) return fail(LAZY_EINVAL, "status is NULL");
  int rc = check_device();
  if (rc) return rc;
  LAZY_CUDA_TRY(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)));
  uint32_t v = 0;
  LAZY_CUDA_TRY(cudaMemcpyFromSymbol(&v, g_status_word, sizeof(v)));
  const uint32_t zero = 0;
  LAZY_CUDA_TRY(cudaMemcpyToSymbol(g_status_word, &zero, sizeof(zero)));
  *status = v;
  return LAZY_OK;
}

}  // extern "C"
