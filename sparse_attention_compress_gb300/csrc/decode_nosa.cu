// The NOSA decode step ([NOSA-Parts] "decoding over only 64 KV blocks"): the decode
// kernels of decode_impl.cuh with CIS-weighted attention and the optional two-stage
// selection (the kept blocks re-ranked by their CIS block score).
#include "decode_impl.cuh"

namespace nsa {

cudaError_t launch_decode_nosa(const DecodeArgs& a, const DecodeLayout& l, cudaStream_t st) {
  return run_decode_all<true>(a, l, st);
}

NSA_STATUS_ACCESSOR(decode_nosa)

}  // namespace nsa
