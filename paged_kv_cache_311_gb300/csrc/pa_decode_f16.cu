// pa_decode_f16.cu -- instantiations of the decode kernel for f16 K/V.
#include "pkv_host.cuh"

namespace pkv {
int launch_decode_f16(const DecodeLaunch &a) { return dispatch_decode<__half>(a); }
}  // namespace pkv
