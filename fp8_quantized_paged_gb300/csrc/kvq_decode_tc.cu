// kvq_decode_tc.cu -- the tensor-core decode kernels (kvq_decode_tc.cuh) of
// the two FP8 formats, compiled in a translation unit of their own so that
// they build in parallel with the other kernels.
#include <mutex>

#include "kvq_decode_tc.cuh"

namespace kvq {
namespace dtc {
template int launch_tc<KVQ_FMT_E4M3>(const DecodeParams&, const CUtensorMap&, const CUtensorMap&,
                                     cudaStream_t);
template int launch_tc<KVQ_FMT_E5M2>(const DecodeParams&, const CUtensorMap&, const CUtensorMap&,
                                     cudaStream_t);

template int choose_clu<KVQ_FMT_E4M3>(int, int, int, int);
template int choose_clu<KVQ_FMT_E5M2>(int, int, int, int);

bool fits_tc(int G, int B, int Hkv) {
  static size_t cap[64];
  static DeviceOnce once;  // the opt-in limit, looked up until a lookup succeeds
  const int dev = current_device();
  if (!once.run(dev, [dev] { return (cap[dev] = smem_optin()) > 0; })) return false;
  return smem_bytes_tc(G, B, Hkv) <= cap[dev];
}
}  // namespace dtc
}  // namespace kvq
