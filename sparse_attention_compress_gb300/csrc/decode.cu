// One decode step: score the newest query against the compressed key cache, pick the
// top-k blocks, attend over them.
//
// [NOSA-Parts] "NOSA-1B core components", how decoding uses only 64 KV blocks: the
// selection picks topk = 64 blocks and the sparse attention runs over those blocks only.
//
// GB300 design.  A decode step has only batch * h_kv independent rows, far fewer than
// the 152 SMs, and the path is HBM bound (compressed keys plus the chosen K/V blocks).
// The whole step is one persistent kernel (cooperative launch, every CTA resident) in two
// phases:
//   scoring: the (row, 32-key unit) space of the compressed keys is cut into one
//      contiguous run per CTA; each warp streams its units through a cp.async ring and
//      writes each unit's (max, sum) per head and its pooled block partials, so the whole
//      phase is one HBM stream with every load issued up front.  A CTA then adds its unit
//      count to each row it touched (arrival counter); the CTA that completes a row folds
//      the partials into block scores, runs a CTA-wide top-k and publishes the row's block
//      list with a release flag;
//   attention: the CTAs take items (row, split of the block list) from a global queue,
//      wait for the row's flag (bounded), stream the split's blocks (four warps, 16-key
//      slices, cp.async rings) and write the split's softmax state; the last split of a
//      row merges them into O.
// A CTA makes its selections before it takes any attention item, so a waiting CTA only
// waits for a selection that a running CTA is making; the gather of the rows selected
// first overlaps the selection of the others.  A memset of the counters and the kernel
// are stream ordered and capture into one CUDA graph.
#include "decode_impl.cuh"

namespace nsa {

static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

DecodeLayout decode_layout(int batch, int max_len, int h, int hkv, int d, int kernel, int stride,
                           int block_size, int k) {
  DecodeLayout l{};
  const int r = h / hkv;
  const int rtiles = (r + 15) / 16;
  const int nc_max = max_len >= kernel ? (max_len - kernel) / stride + 1 : 0;
  l.n_units = nc_max > 0 ? (nc_max + 31) / 32 : 1;  // units of 32 compressed keys
  // about one attention item per resident CTA slot (2 per SM), at most 16 splits
  const int64_t units = (int64_t)batch * hkv * rtiles;
  int ns = (int)(2 * 152 / (units > 0 ? units : 1));
  ns = ns < 1 ? 1 : (ns > 16 ? 16 : ns);
  ns = ns < k ? ns : k;
  const int eps = (k + ns - 1) / ns;  // entries per split; no split is left empty
  l.n_split = (k + eps - 1) / eps;
  size_t off = 0;
  l.z = off;  // per-unit pooled partial sums [batch, hkv, n_units, 8 blocks, r]
  off = align256(off + (size_t)batch * hkv * l.n_units * 8 * r * 4);
  l.unit_ml = off;  // per unit and head (max, sum) [batch, hkv, n_units, r, 2]
  off = align256(off + (size_t)batch * hkv * l.n_units * r * 2 * 4);
  l.idx = off;
  off = align256(off + (size_t)batch * hkv * k * 4);
  l.part_o = off;
  off = align256(off + (size_t)batch * hkv * rtiles * l.n_split * 16 * d * 4);
  l.part_ml = off;
  off = align256(off + (size_t)batch * hkv * rtiles * l.n_split * 16 * 2 * 4);
  l.counters = off;
  // work queue head, score arrivals per row, split arrivals per row, ready flags per row
  l.counter_bytes = (size_t)(1 + (size_t)batch * hkv * (2 + rtiles)) * 4;
  off = align256(off + l.counter_bytes);
  l.total = off;
  return l;
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t st) {
  const DecodeLayout l = decode_layout(a.batch, a.max_len, a.h, a.hkv, a.d, a.kernel, a.stride, a.block_size, a.k);
  if (!a.o || !a.part_o || !a.part_ml || !a.counters || !a.idx) return cudaErrorInvalidValue;
  // queue, arrival counters and ready flags start at zero on every call (a memset)
  cudaError_t e = cudaMemsetAsync(a.counters, 0, l.counter_bytes, st);
  if (e != cudaSuccess) return e;
  if (a.cis) return launch_decode_nosa(a, l, st);
  return run_decode_all<false>(a, l, st);
}

NSA_STATUS_ACCESSOR(decode)

}  // namespace nsa
