// kvq_decode_variant.cu -- the decode kernels of one cache format and head
// size (KVQ_VARIANT_FMT, KVQ_VARIANT_DH, set by the build), so that the
// variants compile in parallel.
#include "kvq_decode.cuh"

#if !defined(KVQ_VARIANT_FMT) || !defined(KVQ_VARIANT_DH)
#error "build with -DKVQ_VARIANT_FMT=<kvq_fmt> -DKVQ_VARIANT_DH=<64|128>"
#endif

namespace kvq {
template int launch<KVQ_VARIANT_FMT, KVQ_VARIANT_DH>(const DecodeParams&, const CUtensorMap&,
                                                     const CUtensorMap&, cudaStream_t);
}  // namespace kvq
