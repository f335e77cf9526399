// kvq_decode_blk.cu -- host side of the whole-block tensor-core decode
// (kvq_decode_blk.cuh): configuration, the shared-memory check and the
// launch, for both FP8 formats.
#include <atomic>
#include <mutex>

#include "kvq_decode_blk.cuh"

namespace kvq {
namespace dtb {

template <int FMT, bool QF8, bool GRID>
static bool configure(size_t maxsmem) {
  auto k = decode_blk_kernel<FMT, QF8, GRID>;
  return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(maxsmem)) == cudaSuccess &&
         cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout,
                              cudaSharedmemCarveoutMaxShared) == cudaSuccess;
}

constexpr int kMaxDev = 64;

// The opt-in shared memory per block of the current device, and whether
// the kernels of format FMT are configured on it.  Both are recorded only
// once they succeed: a failed query or attribute call is retried by the
// next call (its error cleared), not remembered as done.
struct DevState {
  std::mutex mu;
  std::atomic<size_t> optin[kMaxDev];
  std::atomic<bool> conf[2][kMaxDev];
};

static DevState& dev_state() {
  static DevState st;
  return st;
}

static int current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) {
    cudaGetLastError();
    return -1;
  }
  return dev;
}

static size_t optin_of(int dev) {
  DevState& st = dev_state();
  size_t v = st.optin[dev].load(std::memory_order_acquire);
  if (v) return v;
  std::lock_guard<std::mutex> g(st.mu);
  v = st.optin[dev].load(std::memory_order_relaxed);
  if (v) return v;
  int x = 0;
  if (cudaDeviceGetAttribute(&x, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess || x <= 0) {
    cudaGetLastError();
    return 0;
  }
  st.optin[dev].store(static_cast<size_t>(x), std::memory_order_release);
  return static_cast<size_t>(x);
}

template <int FMT>
static bool ensure_configured(int dev) {
  DevState& st = dev_state();
  const int f = FMT == KVQ_FMT_E5M2 ? 1 : 0;
  if (st.conf[f][dev].load(std::memory_order_acquire)) return true;
  const size_t cap = optin_of(dev);
  if (cap == 0) return false;
  std::lock_guard<std::mutex> g(st.mu);
  if (st.conf[f][dev].load(std::memory_order_relaxed)) return true;
  const size_t need = BLay<false>::total(kMaxSeqs, kMaxKvHeads);
  const size_t m = need < cap ? need : cap;
  const bool ok = configure<FMT, false, false>(m) && configure<FMT, true, false>(m) &&
                  configure<FMT, false, true>(m) && configure<FMT, true, true>(m);
  if (!ok) {
    cudaGetLastError();
    return false;
  }
  st.conf[f][dev].store(true, std::memory_order_release);
  return true;
}

bool fits_blk(int B, int Hkv) {
  const int dev = current_device();
  if (dev < 0) return false;
  const size_t cap = optin_of(dev);
  return cap > 0 && BLay<false>::total(B, Hkv) <= cap;
}

template <typename K>
static cudaError_t launch_kernel(K kernel, int grid, size_t smem, cudaStream_t s,
                                 const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreadsB);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, p, tk, tv);
}

template <int FMT>
int launch_blk(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv, bool grid_merge,
               cudaStream_t s) {
  const int dev = current_device();
  if (dev < 0 || !ensure_configured<FMT>(dev)) return KVQ_ERR_CUDA;
  const size_t smem = BLay<false>::total(p.B, p.Hkv);  // the Q-FP8 layout is no larger
  if (smem > optin_of(dev)) return KVQ_ERR_UNSUPPORTED;
  const bool qf8 = p.qs != nullptr;
  cudaError_t e;
  if (grid_merge)
    e = qf8 ? launch_kernel(decode_blk_kernel<FMT, true, true>, p.P, smem, s, p, tk, tv)
            : launch_kernel(decode_blk_kernel<FMT, false, true>, p.P, smem, s, p, tk, tv);
  else
    e = qf8 ? launch_kernel(decode_blk_kernel<FMT, true, false>, p.P, smem, s, p, tk, tv)
            : launch_kernel(decode_blk_kernel<FMT, false, false>, p.P, smem, s, p, tk, tv);
  if (e != cudaSuccess) return KVQ_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

template int launch_blk<KVQ_FMT_E4M3>(const DecodeParams&, const CUtensorMap&, const CUtensorMap&,
                                      bool, cudaStream_t);
template int launch_blk<KVQ_FMT_E5M2>(const DecodeParams&, const CUtensorMap&, const CUtensorMap&,
                                      bool, cudaStream_t);

}  // namespace dtb
}  // namespace kvq
