// ns_muon.cu -- the momentum step of a Muon-style optimizer, the input side
// of ns_muon_update_batched (include/ns.h).
//
// One element-wise pass per matrix: Mom' = mu * Mom + G, rounded to the
// working type and stored back into the momentum buffer; the matrix to
// orthogonalize, X = G + mu * Mom' (Nesterov) or X = Mom', rounded and
// written into the output buffer, where the Newton-Schulz call then works on
// it in place (its last step writes scale * NS(X) there). Arithmetic in fp32;
// 16-byte accesses when the three buffers allow. An output buffer that is the
// gradient buffer itself is allowed: each element is read before it is
// written, by the same thread.
#include <cuda_runtime.h>

#include <algorithm>

#include "ns_device.cuh"

namespace ns {

namespace {

template <int DT>
__device__ __forceinline__ void momentum_elem(const typename Elem<DT>::T &g, typename Elem<DT>::T &m,
                                              typename Elem<DT>::T &x, float mu, int nesterov) {
  const float gf = Elem<DT>::to_f(g);
  const auto ms = Elem<DT>::from_f(fmaf(mu, Elem<DT>::to_f(m), gf));
  m = ms;
  x = nesterov ? Elem<DT>::from_f(fmaf(mu, Elem<DT>::to_f(ms), gf)) : ms;
}

template <int DT>
__global__ void __launch_bounds__(256) ns_momentum_kernel(const __grid_constant__ MomentumParams p) {
  using T = typename Elem<DT>::T;
  constexpr int V = 16 / static_cast<int>(sizeof(T));
  const int k = blockIdx.y;
  const T *g = static_cast<const T *>(p.g[k]);
  T *m = static_cast<T *>(p.mom[k]);
  T *o = static_cast<T *>(p.out[k]);
  const int64_t n = p.numel[k];
  const int64_t first = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const bool vec =
      ((reinterpret_cast<uintptr_t>(g) | reinterpret_cast<uintptr_t>(m) | reinterpret_cast<uintptr_t>(o)) & 15) == 0;
  int64_t done = 0;
  if (vec) {
    const int64_t nv = n / V;
    for (int64_t i = first; i < nv; i += stride) {
      uint4 gw = *reinterpret_cast<const uint4 *>(g + i * V);
      uint4 mw = *reinterpret_cast<const uint4 *>(m + i * V);
      uint4 xw;
      const T *ge = reinterpret_cast<const T *>(&gw);
      T *me = reinterpret_cast<T *>(&mw);
      T *xe = reinterpret_cast<T *>(&xw);
#pragma unroll
      for (int e = 0; e < V; ++e) momentum_elem<DT>(ge[e], me[e], xe[e], p.mu, p.nesterov);
      if (in_bounds(m + i * V, 16, m, n * sizeof(T), p.status)) *reinterpret_cast<uint4 *>(m + i * V) = mw;
      if (in_bounds(o + i * V, 16, o, n * sizeof(T), p.status)) *reinterpret_cast<uint4 *>(o + i * V) = xw;
    }
    done = nv * V;
  }
  for (int64_t i = done + first; i < n; i += stride) {
    T mv = m[i], xv;
    momentum_elem<DT>(g[i], mv, xv, p.mu, p.nesterov);
    if (in_bounds(m + i, sizeof(T), m, n * sizeof(T), p.status)) m[i] = mv;
    if (in_bounds(o + i, sizeof(T), o, n * sizeof(T), p.status)) o[i] = xv;
  }
}

// Self-test of the debug bounds checks: one thread asks whether a 16-byte
// store one past the end of a 4-byte buffer is in bounds. Nothing is stored
// either way; a debug build records kStatusBounds.
__global__ void ns_bounds_probe_kernel(int *status, const void *base) {
  const uint8_t *past = static_cast<const uint8_t *>(base) + 4;
  (void)in_bounds(past, 16, base, 4, status);
}

}  // namespace

int launch_bounds_probe(int *status, const void *base, cudaStream_t s) {
  ns_bounds_probe_kernel<<<1, 1, 0, s>>>(status, base);
  count_launch();
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

int launch_momentum(const MomentumParams &p, int dtype, int sms, cudaStream_t s) {
  if (p.count <= 0) return 0;
  int64_t most = 0;
  for (int k = 0; k < p.count; ++k) most = std::max(most, p.numel[k]);
  const int per_block = 256 * 8 * 4;  // elements a block covers in four 16-byte rounds (bf16)
  const int64_t want = (most + per_block - 1) / per_block;
  const int bx = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(want, 4 * sms)));
  const dim3 grid(bx, p.count, 1);
  if (dtype == kBF16)
    ns_momentum_kernel<kBF16><<<grid, 256, 0, s>>>(p);
  else
    ns_momentum_kernel<kF32><<<grid, 256, 0, s>>>(p);
  count_launch();
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace ns
