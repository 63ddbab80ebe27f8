// ns_simt.cu -- CUDA-core kernels of libns:
//   * per-matrix Frobenius norm (partial sums) and non-zero extent (fp32 path),
//   * the per-matrix scale from the bf16 norm pass's tile sums,
//   * preparation: normalise by ||Y||_F + eps, round to the working type and
//     write both orientations W and W^T,
//   * the shared-memory resident kernel that runs every step of a small
//     matrix inside one CTA,
//   * the fp32 tiled GEMM phases (gram / square / apply) for large fp32
//     matrices.
// The bf16 norm pass lives in ns_norm.cu, the bf16 tensor-core phases in
// ns_tc.cu.
#include <cuda_runtime.h>

#include <algorithm>

#include "ns_device.cuh"

namespace ns {

// ============================================================== norm + extent
// Grid kNormBlocks * nmats. Block b of matrix i visits rows b, b+kNormBlocks,
// ... in a fixed order, so the partial sums are the same on every run. It also
// records the largest row and column index that holds a non-zero, in the
// caller's orientation; zero rows/columns beyond them stay zero through every
// step (the first page's "Fix" section) and are skipped by the GEMM phases.
template <int DT>
__global__ void __launch_bounds__(256) ns_norm_kernel(PrepParams p) {
  using T = typename Elem<DT>::T;
  const int mat = blockIdx.x / kNormBlocks;
  const int blk = blockIdx.x % kNormBlocks;
  const MatDesc &d = p.mats[mat];
  const T *y = static_cast<const T *>(d.user);
  const int M = d.M, N = d.N;
  constexpr int VEC = 16 / sizeof(T);
  const bool vec = (N % VEC == 0) && ((reinterpret_cast<uintptr_t>(y) & 15) == 0);

  float acc = 0.f;
  int rmax = -1, cmax = -1;
  for (int r = blk; r < M; r += kNormBlocks) {
    const T *row = y + static_cast<size_t>(r) * N;
    bool any = false;
    if (vec) {
      const uint4 *row4 = reinterpret_cast<const uint4 *>(row);
      for (int c4 = threadIdx.x; c4 < N / VEC; c4 += blockDim.x) {
        uint4 raw = __ldg(row4 + c4);
        const T *e = reinterpret_cast<const T *>(&raw);
#pragma unroll
        for (int u = 0; u < VEC; ++u) {
          const float v = Elem<DT>::to_f(e[u]);
          acc = fmaf(v, v, acc);
          if (v != 0.f) {
            any = true;
            cmax = max(cmax, c4 * VEC + u);
          }
        }
      }
    } else {
      for (int c = threadIdx.x; c < N; c += blockDim.x) {
        const float v = Elem<DT>::load(row + c);
        acc = fmaf(v, v, acc);
        if (v != 0.f) {
          any = true;
          cmax = max(cmax, c);
        }
      }
    }
    if (any) rmax = r;
  }

  __shared__ float s_sum[8];
  __shared__ int s_r[8], s_c[8];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  acc = warp_sum(acc);
  rmax = warp_max(rmax);
  cmax = warp_max(cmax);
  if (lane == 0) {
    s_sum[warp] = acc;
    s_r[warp] = rmax;
    s_c[warp] = cmax;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    int rr = -1, cc = -1;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) {
      t += s_sum[w];
      rr = max(rr, s_r[w]);
      cc = max(cc, s_c[w]);
    }
    p.partials[mat * kNormBlocks + blk] = t;
    if (rr >= 0) atomicMax(&p.ext[2 * mat + 0], rr + 1);
    if (cc >= 0) atomicMax(&p.ext[2 * mat + 1], cc + 1);
  }
}

int launch_norm(const PrepParams &p, cudaStream_t s) {
  if (p.nmats <= 0) return 0;
  const unsigned grid = static_cast<unsigned>(kNormBlocks) * static_cast<unsigned>(p.nmats);
  if (p.dtype == kBF16)
    ns_norm_kernel<kBF16><<<grid, 256, 0, s>>>(p);
  else
    ns_norm_kernel<kF32><<<grid, 256, 0, s>>>(p);
  count_launch();
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

// ============================================================== preparation
// One block per 64x64 tile of the caller's Y. Every block sums the
// matrix's kNormBlocks partials in the same fixed order, so all blocks agree
// on s = ||Y||_F. It writes y * (1 / (s + eps)), rounded to the working type, into
// W and W^T (or back into Y when no step follows). When Y's rows are 16-byte
// aligned the tile moves in 16-byte vectors; the transposed copy goes through
// shared memory so both writes are row-contiguous.
template <int DT>
__global__ void __launch_bounds__(256) ns_prep_kernel(PrepParams p) {
  using T = typename Elem<DT>::T;
  constexpr int V = 16 / sizeof(T);                 // elements per 16-byte vector
  constexpr int CPR = kPrepTile / V;                // vectors per tile row
  constexpr int PER = kPrepTile * kPrepTile / V / 256;  // vectors per thread
  const int bid = blockIdx.x;
  int lo = 0, hi = p.nmats;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (p.tile_prefix[mid] <= bid) lo = mid; else hi = mid;
  }
  const int mat = lo;
  const MatDesc &d = p.mats[mat];
  const int M = d.M, N = d.N;
  const int local = bid - p.tile_prefix[mat];
  const int tcols = (N + kPrepTile - 1) / kPrepTile;
  const int r0 = (local / tcols) * kPrepTile, c0 = (local % tcols) * kPrepTile;
  const T *y = static_cast<const T *>(d.user);
  const bool vec = (N % V == 0) && ((reinterpret_cast<uintptr_t>(y) & 15) == 0);

  __shared__ float s_denom;  // reciprocal of ||Y||_F + eps
  __shared__ float tile[kPrepTile][kPrepTile + 1];
  const int tid = threadIdx.x;

  // raw loads first: they do not depend on the norm
  uint4 raw[PER];
  if (vec) {
#pragma unroll
    for (int k = 0; k < PER; ++k) {
      const int q = tid + k * 256, rr = q / CPR, cv = q % CPR;
      const int r = r0 + rr, c = c0 + cv * V;
      raw[k] = make_uint4(0, 0, 0, 0);
      if (r < M && c < N) raw[k] = __ldg(reinterpret_cast<const uint4 *>(y + static_cast<size_t>(r) * N + c));
    }
  }
  if (tid < 32) {
    float v = 0.f;
    for (int i = tid; i < kNormBlocks; i += 32) v += p.partials[mat * kNormBlocks + i];
    v = warp_sum(v);
    if (tid == 0) s_denom = 1.0f / (sqrtf(v) + p.eps);  // 1 / (||Y||_F + eps)
  }
  __syncthreads();
  const float inv = s_denom;
  if (vec) {
#pragma unroll
    for (int k = 0; k < PER; ++k) {
      const int q = tid + k * 256, rr = q / CPR, cv = q % CPR;
      const T *e = reinterpret_cast<const T *>(&raw[k]);
#pragma unroll
      for (int u = 0; u < V; ++u) tile[rr][cv * V + u] = Elem<DT>::to_f(e[u]) * inv;
    }
  } else {
    for (int e = tid; e < kPrepTile * kPrepTile; e += 256) {
      const int rr = e / kPrepTile, cc = e % kPrepTile;
      const int r = r0 + rr, c = c0 + cc;
      float v = 0.f;
      if (r < M && c < N) v = Elem<DT>::load(y + static_cast<size_t>(r) * N + c) * inv;
      tile[rr][cc] = v;
    }
  }
  __syncthreads();

  // writes: destination rows are 16-byte aligned (workspace pitches are
  // multiples of 8 elements; the caller's rows when `vec`)
  auto write_tile = [&](T *dst, int pitch, bool flip, int rows, int cols, bool dst_vec) {
    // the tile as seen by the destination: rows x cols = (flip ? 64 cols of Y : 64 rows of Y)
    const int R0 = flip ? c0 : r0, C0 = flip ? r0 : c0;
#pragma unroll
    for (int k = 0; k < PER; ++k) {
      const int q = tid + k * 256, rr = q / CPR, cv = q % CPR;
      const int R = R0 + rr, C = C0 + cv * V;
      if (R >= rows || C >= cols) continue;
      T *out = dst + static_cast<size_t>(R) * pitch + C;
      if (dst_vec && C + V <= cols) {
        uint4 w;
        T *we = reinterpret_cast<T *>(&w);
#pragma unroll
        for (int u = 0; u < V; ++u) we[u] = Elem<DT>::from_f(flip ? tile[cv * V + u][rr] : tile[rr][cv * V + u]);
        *reinterpret_cast<uint4 *>(out) = w;
      } else {
        for (int u = 0; u < V && C + u < cols; ++u)
          out[u] = Elem<DT>::from_f(flip ? tile[cv * V + u][rr] : tile[rr][cv * V + u]);
      }
    }
  };

  if (p.to_user) {
    write_tile(static_cast<T *>(d.user), N, false, M, N, vec);
    return;
  }
  // same orientation as Y: W when not transposed, W^T when transposed
  T *same = static_cast<T *>(d.transposed ? d.xt[0] : d.x);
  const int same_pitch = d.transposed ? d.pm : d.pn;
  // transposed orientation: W^T when not transposed, W when transposed
  T *flip = static_cast<T *>(d.transposed ? d.x : d.xt[0]);
  const int flip_pitch = d.transposed ? d.pn : d.pm;
  write_tile(same, same_pitch, false, M, N, true);
  write_tile(flip, flip_pitch, true, N, M, true);
}

int launch_prep(const PrepParams &p, int total_tiles, cudaStream_t s) {
  if (total_tiles <= 0) return 0;
  if (p.dtype == kBF16)
    ns_prep_kernel<kBF16><<<total_tiles, 256, 0, s>>>(p);
  else
    ns_prep_kernel<kF32><<<total_tiles, 256, 0, s>>>(p);
  count_launch();
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

// One block per matrix: the tile partial sums of the matrix in a fixed order
// (strided per thread, then a fixed tree) give r = 1 / (||Y||_F + eps).
__global__ void __launch_bounds__(256) ns_norm_finish_kernel(PrepParams p) {
  const int mat = blockIdx.x;
  const int t0 = p.tile_prefix[mat], t1 = p.tile_prefix[mat + 1];
  float v = 0.f;
  for (int i = t0 + static_cast<int>(threadIdx.x); i < t1; i += 256) v += p.tile_partials[i];
  __shared__ float s_sum[8];
  v = warp_sum(v);
  if ((threadIdx.x & 31) == 0) s_sum[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int w = 0; w < 8; ++w) t += s_sum[w];
    p.rscale[mat] = 1.0f / (sqrtf(t) + p.eps);
  }
}

int launch_norm_finish(const PrepParams &p, cudaStream_t s) {
  if (p.nmats <= 0) return 0;
  ns_norm_finish_kernel<<<p.nmats, 256, 0, s>>>(p);
  count_launch();
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

// ============================================================== resident
// One CTA of 256 threads runs the whole method for one small matrix
// (m <= 64) held in shared memory: W (mp x np, working type, zero padded to
// multiples of 4), A and B (fp32). Y is read once and written once. All work
// is on 4 x 4 register blocks with a fixed assignment and fixed reduction
// order, so results repeat bit for bit:
//   gram    upper-triangle blocks of A = W W^T; when there are few blocks the
//           contraction over n is split into S slices whose partial blocks
//           are summed in slice order;
//   square  upper-triangle blocks of B = b A + c A A (A, B kept symmetric);
//   apply   W' = a W + B W in column panels: every thread computes one 4 x 4
//           block of the panel, then the panel is written back in place.
// Only the non-zero block [0, meff) x [0, neff) is iterated on.
namespace {
constexpr int kResThreads = 256;
constexpr int kResPartials = kResThreads * 16;  // floats of the split-gram scratch

__host__ __device__ inline size_t res_align16(size_t v) { return (v + 15) & ~size_t(15); }

struct ResLayout {
  int mp, np, ap;
  size_t off_a, off_b, off_part, total;
  __host__ __device__ ResLayout(int m, int n, int elt) {
    mp = (m + 3) & ~3;
    np = (n + 3) & ~3;
    ap = mp + 1;
    off_a = res_align16(static_cast<size_t>(mp) * np * elt);
    off_b = res_align16(off_a + static_cast<size_t>(mp) * ap * 4);
    off_part = res_align16(off_b + static_cast<size_t>(mp) * ap * 4);
    total = off_part + static_cast<size_t>(kResPartials) * 4;
  }
};

// (bi, bj), bi <= bj, of upper-triangle block number b (row-major order)
__device__ __forceinline__ void upper_block(int b, int mb, int &bi, int &bj) {
  bi = 0;
  while (b >= mb - bi) {
    b -= mb - bi;
    ++bi;
  }
  bj = bi + b;
}
}  // namespace

int resident_smem_bytes(int m, int n, int dtype) {
  const ResLayout L(m, n, dtype == kBF16 ? 2 : 4);
  return L.total > (size_t(1) << 30) ? (1 << 30) : static_cast<int>(L.total);
}

template <int DT>
__global__ void __launch_bounds__(kResThreads, 1) ns_resident_kernel(ResParams p) {
  using T = typename Elem<DT>::T;
  extern __shared__ __align__(16) uint8_t smem[];
  const ResDesc d = p.mats[blockIdx.x];
  const int M = d.M, N = d.N, m = d.m, n = d.n, tr = d.transposed;
  const ResLayout L(m, n, sizeof(T));
  const int np = L.np, ap = L.ap;
  T *xs = reinterpret_cast<T *>(smem);
  float *as = reinterpret_cast<float *>(smem + L.off_a);
  float *bs = reinterpret_cast<float *>(smem + L.off_b);
  float *part = reinterpret_cast<float *>(smem + L.off_part);
  T *y = static_cast<T *>(d.user);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  constexpr int NW = kResThreads / 32;

  __shared__ float s_sum[NW];
  __shared__ int s_r[NW], s_c[NW];
  __shared__ float s_denom;  // reciprocal of ||Y||_F + eps
  __shared__ int s_meff, s_neff;

  // 1. zero the padded working copy, then load Y into it (oriented as W),
  //    with the sum of squares and the non-zero extent
  for (int e = tid; e < L.mp * np; e += kResThreads) xs[e] = Elem<DT>::from_f(0.f);
  __syncthreads();
  float acc = 0.f;
  int rmax = -1, cmax = -1;
  for (int r = warp; r < M; r += NW) {
    const T *row = y + static_cast<size_t>(r) * N;
    bool any = false;
#pragma unroll 4
    for (int c = lane; c < N; c += 32) {
      const T v = row[c];
      const float f = Elem<DT>::to_f(v);
      acc = fmaf(f, f, acc);
      if (f != 0.f) {
        any = true;
        cmax = max(cmax, c);
      }
      if (tr) xs[c * np + r] = v; else xs[r * np + c] = v;
    }
    if (any) rmax = r;
  }
  acc = warp_sum(acc);
  rmax = warp_max(rmax);
  cmax = warp_max(cmax);
  if (lane == 0) {
    s_sum[warp] = acc;
    s_r[warp] = rmax;
    s_c[warp] = cmax;
  }
  __syncthreads();
  if (tid == 0) {
    float t = 0.f;
    int rr = -1, cc = -1;
    for (int w = 0; w < NW; ++w) {
      t += s_sum[w];
      rr = max(rr, s_r[w]);
      cc = max(cc, s_c[w]);
    }
    s_denom = 1.0f / (sqrtf(t) + p.eps);  // 1 / (||Y||_F + eps)
    s_meff = tr ? cc + 1 : rr + 1;
    s_neff = tr ? rr + 1 : cc + 1;
  }
  __syncthreads();
  const float inv = s_denom;
  const int meff = s_meff, neff = s_neff;

  // 2. normalise (zeros stay zero)
  for (int e = tid; e < L.mp * np; e += kResThreads)
    xs[e] = Elem<DT>::from_f(Elem<DT>::to_f(xs[e]) * inv);
  __syncthreads();

  // 3. iterate on the non-zero block
  const int mb = (meff + 3) / 4;          // 4-row blocks holding non-zero rows
  const int nblk = mb * (mb + 1) / 2;     // upper-triangle blocks
  const int S = nblk > 0 ? max(1, min(kResThreads / max(nblk, 1), neff)) : 1;  // gram slices
  const int kslice = (neff + S - 1) / S;
  const int panel = 4 * (kResThreads / max(mb, 1));  // apply: columns per panel
  for (int step = 0; step < p.steps && meff > 0; ++step) {
    const float *co = p.coef[p.ncoef == 1 ? 0 : step];
    const float ca = co[0], cb = co[1], cc = co[2];
    // ---- gram: partial 4x4 blocks over k-slices
    if (tid < nblk * S) {
      const int b = tid / S, sl = tid % S;
      int bi, bj;
      upper_block(b, mb, bi, bj);
      const int k0 = sl * kslice, k1 = min(neff, k0 + kslice);
      float c4[4][4] = {};
      for (int k = k0; k < k1; ++k) {
        float xa[4], xb[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          xa[u] = Elem<DT>::to_f(xs[(4 * bi + u) * np + k]);
          xb[u] = Elem<DT>::to_f(xs[(4 * bj + u) * np + k]);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
          for (int v = 0; v < 4; ++v) c4[u][v] = fmaf(xa[u], xb[v], c4[u][v]);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int v = 0; v < 4; ++v) part[(sl * nblk + b) * 16 + u * 4 + v] = c4[u][v];
    }
    __syncthreads();
    // ---- sum the slices in order into A (both triangles)
    for (int e = tid; e < nblk * 16; e += kResThreads) {
      const int b = e >> 4, u = (e >> 2) & 3, v = e & 3;
      int bi, bj;
      upper_block(b, mb, bi, bj);
      float sum = 0.f;
      for (int sl = 0; sl < S; ++sl) sum += part[(sl * nblk + b) * 16 + u * 4 + v];
      const int i = 4 * bi + u, j = 4 * bj + v;
      if (bi < bj || u <= v) {
        as[i * ap + j] = sum;
        as[j * ap + i] = sum;
      }
    }
    __syncthreads();
    // ---- square: B = b A + c A A on upper blocks (symmetric, so both triangles)
    for (int b = tid; b < nblk; b += kResThreads) {
      int bi, bj;
      upper_block(b, mb, bi, bj);
      float c4[4][4] = {};
      for (int k = 0; k < meff; ++k) {
        float ar[4], ac[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          ar[u] = as[(4 * bi + u) * ap + k];
          ac[u] = as[k * ap + 4 * bj + u];
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
          for (int v = 0; v < 4; ++v) c4[u][v] = fmaf(ar[u], ac[v], c4[u][v]);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const int i = 4 * bi + u, j = 4 * bj + v;
          const float val = cb * as[i * ap + j] + cc * c4[u][v];
          bs[i * ap + j] = val;
          bs[j * ap + i] = val;
        }
    }
    __syncthreads();
    // ---- apply: W' = a W + B W, one column panel at a time
    for (int c0 = 0; c0 < neff; c0 += panel) {
      const int rb = tid % mb, cb = tid / mb;
      const int j0 = c0 + 4 * cb;
      const bool active = tid < mb * (panel / 4) && j0 < neff;
      float o4[4][4] = {};
      if (active) {
        for (int k = 0; k < meff; ++k) {
          float br[4], xr[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            br[u] = bs[(4 * rb + u) * ap + k];
            xr[u] = Elem<DT>::to_f(xs[k * np + j0 + u]);
          }
#pragma unroll
          for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int v = 0; v < 4; ++v) o4[u][v] = fmaf(br[u], xr[v], o4[u][v]);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
          for (int v = 0; v < 4; ++v)
            o4[u][v] = ca * Elem<DT>::to_f(xs[(4 * rb + u) * np + j0 + v]) + o4[u][v];
      }
      __syncthreads();  // every read of this panel happened
      if (active) {
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
          for (int v = 0; v < 4; ++v) xs[(4 * rb + u) * np + j0 + v] = Elem<DT>::from_f(o4[u][v]);
      }
      __syncthreads();
    }
  }

  // 4. write back in the caller's orientation
  for (int r = warp; r < M; r += NW) {
    T *row = y + static_cast<size_t>(r) * N;
#pragma unroll 4
    for (int c = lane; c < N; c += 32) row[c] = tr ? xs[c * np + r] : xs[r * np + c];
  }
}

template <int DT>
static int launch_resident_t(const ResParams &p, int smem, cudaStream_t s) {
  auto k = ns_resident_kernel<DT>;
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) return -1;
  k<<<p.nmats, kResThreads, smem, s>>>(p);
  count_launch();
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

int launch_resident(const ResParams &p, int maxm, int smem, cudaStream_t s) {
  (void)maxm;
  if (p.nmats <= 0) return 0;
  if (p.dtype == kBF16) return launch_resident_t<kBF16>(p, smem, s);
  return launch_resident_t<kF32>(p, smem, s);
}

// ============================================================== fp32 GEMM phases
// One 64x64 output tile per block, 256 threads with 4x4 outputs each,
// C[r, c] = sum_k P[r, k] Q[c, k] over k < K (both operands K-contiguous).
//   phase 0 (gram)   P = Q = W           K = n   -> A (upper + mirror)
//   phase 1 (square) P = Q = A           K = m   -> B = b A + c C (upper + mirror)
//   phase 2 (apply)  P = W^T, Q = B      K = m   -> W' = a W + (B W): W'^T and W,
//                                                   or the caller's Y on the last step
template <int PHASE>
__global__ void __launch_bounds__(256) ns_simt_gemm_kernel(PhaseParams p) {
  const Tile tl = p.tiles[blockIdx.x];
  const MatDesc &d = p.mats[tl.mat];
  const int e0 = p.ext[2 * tl.mat], e1 = p.ext[2 * tl.mat + 1];
  const int meff = d.transposed ? e1 : e0, neff = d.transposed ? e0 : e1;
  const int m = d.m, n = d.n, pm = d.pm, pn = d.pn;
  const int rows_eff = PHASE == 2 ? neff : meff;
  if (tl.row0 >= rows_eff || tl.col0 >= meff) return;
  const int K = PHASE == 0 ? neff : meff;
  const int rows = PHASE == 2 ? n : m;
  const int cols = m;
  const int cur = p.step & 1;
  const float *P = static_cast<const float *>(PHASE == 0 ? d.x : PHASE == 1 ? d.a : d.xt[cur]);
  const float *Q = static_cast<const float *>(PHASE == 0 ? d.x : PHASE == 1 ? d.a : d.b);
  const int pitch_p = PHASE == 0 ? pn : pm;
  const int pitch_q = PHASE == 0 ? pn : pm;

  __shared__ float Ps[16][kSimtBM + 4];
  __shared__ float Qs[16][kSimtBN + 4];
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += 16) {
    for (int e = tid; e < kSimtBM * 16; e += 256) {
      const int rr = e >> 4, kk = e & 15;
      const int r = tl.row0 + rr, k = k0 + kk;
      Ps[kk][rr] = (r < rows && k < K) ? P[static_cast<size_t>(r) * pitch_p + k] : 0.f;
      const int c = tl.col0 + rr;
      Qs[kk][rr] = (c < cols && k < K) ? Q[static_cast<size_t>(c) * pitch_q + k] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        a[u] = Ps[kk][ty * 4 + u];
        b[u] = Qs[kk][tx * 4 + u];
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int v = 0; v < 4; ++v) acc[u][v] = fmaf(a[u], b[v], acc[u][v]);
    }
    __syncthreads();
  }

#pragma unroll
  for (int u = 0; u < 4; ++u) {
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const int r = tl.row0 + ty * 4 + u, c = tl.col0 + tx * 4 + v;
      const float val = acc[u][v];
      if (PHASE == 0 || PHASE == 1) {
        if (r < m && c < m && r <= c) {
          float out = val;
          float *dst = static_cast<float *>(PHASE == 0 ? d.a : d.b);
          if (PHASE == 1) out = p.cb * static_cast<const float *>(d.a)[static_cast<size_t>(r) * pm + c] + p.cc * val;
          dst[static_cast<size_t>(r) * pm + c] = out;
          dst[static_cast<size_t>(c) * pm + r] = out;
        }
      } else {
        if (r < n && c < m) {
          const float *xt = static_cast<const float *>(d.xt[cur]);
          const float out = p.ca * xt[static_cast<size_t>(r) * pm + c] + val;
          if (!p.final_step) {
            static_cast<float *>(d.xt[cur ^ 1])[static_cast<size_t>(r) * pm + c] = out;
            static_cast<float *>(d.x)[static_cast<size_t>(c) * pn + r] = out;
          } else {
            float *u = static_cast<float *>(d.user);
            if (d.transposed) u[static_cast<size_t>(r) * d.N + c] = out;
            else u[static_cast<size_t>(c) * d.N + r] = out;
          }
        }
      }
    }
  }
}

int launch_simt_phase(int phase, const PhaseParams &p, cudaStream_t s) {
  if (p.ntiles <= 0) return 0;
  if (phase == 0) ns_simt_gemm_kernel<0><<<p.ntiles, 256, 0, s>>>(p);
  else if (phase == 1) ns_simt_gemm_kernel<1><<<p.ntiles, 256, 0, s>>>(p);
  else ns_simt_gemm_kernel<2><<<p.ntiles, 256, 0, s>>>(p);
  count_launch();
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace ns
