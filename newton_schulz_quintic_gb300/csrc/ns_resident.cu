// ns_resident.cu -- small matrices (m <= 64) done entirely in shared memory.
//
// Each matrix is worked on by a cluster of C CTAs (C = 1, 2, 4 or 8, chosen
// from the matrix's shape alone, so a matrix gets the same bits in any batch)
// that split W's columns: CTA c holds columns [c*ns, (c+1)*ns) of W (m x n,
// W = Y, or Y^T when M > N) for the whole call. The method's structure makes
// the columns independent except through A = W W^T, which is a sum over
// columns:
//   norm    every CTA sums the squares of its slice (W-row-major order, fixed
//           tree) and finds its non-zero extent; the cluster adds the C sums
//           in rank order and takes the largest row extent;
//   gram    every CTA forms the partial W_c W_c^T over its own columns (upper
//           4 x 4 blocks; the contraction split into slices summed in slice
//           order) and stores it into its slot of every CTA's receive buffer
//           (remote stores through distributed shared memory); after one
//           cluster barrier every CTA adds the C slots in rank order (A, both
//           triangles);
//   square  B = b A + c A A, by every CTA for itself (m <= 64);
//   apply   W_c' = a W_c + B W_c on the CTA's own columns, in column panels
//           written back in place.
// The receive buffers are double-buffered across steps, so one cluster
// barrier per step orders every exchange, and nothing waits on a remote load. The first step folds the normalisation in
// (A = r^2 sum of partials, W_1 = r (a W + B W), r = 1 / (||Y||_F + eps)), so
// the normalised input is never rounded; every later iterate is stored in the
// working type (bf16 rounding to nearest even between steps, as on the
// tensor-core path). Y is read once and written once, with 16-byte accesses
// where its rows allow, and only inside the non-zero extent: padded rows and
// columns are never written. Every reduction has a fixed order, and W is
// held in W's orientation, so Y and Y^T give bit-identical results.
#include <cuda_runtime.h>

#include <algorithm>

#include "ns_device.cuh"

namespace ns {

namespace {

constexpr int kResThreads = 256;
constexpr int kResPartials = kResThreads * 16;  // floats of the split-gram scratch

__host__ __device__ inline size_t res_align16(size_t v) { return (v + 15) & ~size_t(15); }

// Shared-memory layout of one CTA: W slice (mp x ld, working type), A, B
// and the two partial-gram buffers (mp x ap, fp32), the split-gram scratch.
struct ResLayout {
  int mp, ld, ap;
  int nent;  // entries of the upper 4 x 4 blocks of an mp x mp matrix
  size_t off_a, off_b, off_r, off_part, total;
  __host__ __device__ ResLayout(int m, int ns, int elt, int C) {
    const int vec = 16 / elt;  // elements per 16 bytes
    mp = (m + 3) & ~3;
    ld = ns;
    if ((ld / vec) % 2 == 0) ld += vec;  // an odd number of 16-byte units: rows spread over banks
    ap = mp;  // fp32 rows of A, B, P: 16-byte aligned, an odd number of 16-byte units
    if ((ap / 4) % 2 == 0) ap += 4;
    off_a = res_align16(static_cast<size_t>(mp) * ld * elt);
    off_b = res_align16(off_a + static_cast<size_t>(mp) * ap * 4);
    nent = (mp / 4) * (mp / 4 + 1) / 2 * 16;
    // receive slots of the partial Grams: two step parities x C source ranks
    off_r = res_align16(off_b + static_cast<size_t>(mp) * ap * 4);
    off_part = res_align16(off_r + static_cast<size_t>(2) * C * nent * 4);
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

// 8 consecutive elements of a shared-memory row as fp32 (16-byte aligned)
__device__ __forceinline__ void ld8(const __nv_bfloat16 *p, float (&f)[8]) {
  const uint4 w = *reinterpret_cast<const uint4 *>(p);
  const uint32_t q[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    f[2 * k] = __uint_as_float(q[k] << 16);
    f[2 * k + 1] = __uint_as_float(q[k] & 0xFFFF0000u);
  }
}
__device__ __forceinline__ void ld8(const float *p, float (&f)[8]) {
  const float4 a = *reinterpret_cast<const float4 *>(p), b = *reinterpret_cast<const float4 *>(p + 4);
  f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
  f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}
// 4 consecutive elements (8- or 16-byte aligned)
__device__ __forceinline__ void ld4(const __nv_bfloat16 *p, float (&f)[4]) {
  const uint2 w = *reinterpret_cast<const uint2 *>(p);
  f[0] = __uint_as_float(w.x << 16);
  f[1] = __uint_as_float(w.x & 0xFFFF0000u);
  f[2] = __uint_as_float(w.y << 16);
  f[3] = __uint_as_float(w.y & 0xFFFF0000u);
}
__device__ __forceinline__ void ld4(const float *p, float (&f)[4]) {
  const float4 a = *reinterpret_cast<const float4 *>(p);
  f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
}

__device__ __forceinline__ float ld_cluster_f32(const float *local, int rank) {
  return __uint_as_float(ld_shared_cluster_u32(mapa_shared(smem_u32(local), static_cast<uint32_t>(rank))));
}
__device__ __forceinline__ int ld_cluster_i32(const int *local, int rank) {
  return static_cast<int>(ld_shared_cluster_u32(mapa_shared(smem_u32(local), static_cast<uint32_t>(rank))));
}
__device__ __forceinline__ void st_cluster_f32(float *local, int rank, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(mapa_shared(smem_u32(local), static_cast<uint32_t>(rank))),
               "f"(v)
               : "memory");
}

// Sum over the cluster's ranks, in rank order, of the float at `local`'s
// offset in each CTA: the C remote loads are issued together, then added.
template <int C>
__device__ __forceinline__ float cluster_sum(const float *local) {
  float v[C];
#pragma unroll
  for (int c = 0; c < C; ++c) v[c] = C > 1 ? ld_cluster_f32(local, c) : *local;
  float t = 0.f;
#pragma unroll
  for (int c = 0; c < C; ++c) t += v[c];
  return t;
}

// Barrier over the matrix's CTAs: the cluster, or just this CTA when C = 1.
__device__ __forceinline__ void res_sync(int C) {
  if (C > 1) cluster_sync(); else __syncthreads();
}

}  // namespace

int resident_smem_bytes(int m, int ns, int dtype, int cluster) {
  const ResLayout L(m, ns, dtype == kBF16 ? 2 : 4, cluster);
  return L.total > (size_t(1) << 30) ? (1 << 30) : static_cast<int>(L.total);
}

// CTAs per matrix: about 2^17 multiply-adds of one step's gram and apply per
// CTA, a power of two up to 8, and slices at least 8 columns wide.
int resident_cluster(int m, int n) {
  const int64_t mp = (m + 3) & ~3;
  const int64_t work = mp * mp * n;
  int c = 1;
  while (c < 8 && work > (int64_t(1) << 17) * c && n >= 16 * c) c *= 2;
  return c;
}

// Slice width of a matrix split over c CTAs: a multiple of 8 columns.
int resident_slice(int n, int c) { return ((n + c - 1) / c + 7) & ~7; }

namespace {

template <int DT, int C>
__global__ void __launch_bounds__(kResThreads, 1) ns_resident_kernel(const __grid_constant__ ResParams p) {
  using T = typename Elem<DT>::T;
  constexpr int V = 16 / static_cast<int>(sizeof(T));
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ float s_wsum[kResThreads / 32];
  __shared__ int s_wr[kResThreads / 32], s_wc[kResThreads / 32];
  __shared__ float s_sum;       // this CTA's sum of squares (read by the cluster)
  __shared__ int s_rows;        // this CTA's non-zero W rows (read by the cluster)
  __shared__ float s_r;
  __shared__ int s_meff, s_nse;

  const int rank = C > 1 ? static_cast<int>(cluster_ctarank()) : 0;
  const ResDesc d = p.mats[blockIdx.x / C];
  const int M = d.M, N = d.N, m = d.m, n = d.n, tr = d.transposed, ns = d.ns;
  const int c0 = rank * ns;                        // first W column of this CTA
  const int ncols = max(0, min(ns, n - c0));       // W columns held here
  const ResLayout L(m, ns, sizeof(T), C);
  const int ld = L.ld, ap = L.ap, mp = L.mp;
  T *w = reinterpret_cast<T *>(smem);
  float *A = reinterpret_cast<float *>(smem + L.off_a);
  float *B = reinterpret_cast<float *>(smem + L.off_b);
  float *R = reinterpret_cast<float *>(smem + L.off_r);  // R[(parity * C + source rank) * nent + entry]
  const int nent = L.nent;
  float *part = reinterpret_cast<float *>(smem + L.off_part);
  T *y = static_cast<T *>(d.user);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool yvec = (reinterpret_cast<uintptr_t>(y) % 16 == 0) && (N % V == 0);

  // 1. the slice of W, zero padded: rows [0, mp), columns [0, ld)
  for (int e = tid; e < mp * ld / V; e += kResThreads) reinterpret_cast<uint4 *>(w)[e] = make_uint4(0, 0, 0, 0);
  __syncthreads();
  if (!tr) {  // W = Y: row i of the slice is Y[i, c0 .. c0 + ncols)
    if (yvec) {
      const int per = ncols / V;
      for (int e = tid; e < M * per; e += kResThreads) {
        const int i = e / per, j = (e - i * per) * V;
        *reinterpret_cast<uint4 *>(w + i * ld + j) =
            __ldg(reinterpret_cast<const uint4 *>(y + static_cast<size_t>(i) * N + c0 + j));
      }
    } else {
      for (int e = tid; e < M * ncols; e += kResThreads) {
        const int i = e / ncols, j = e - i * ncols;
        w[i * ld + j] = y[static_cast<size_t>(i) * N + c0 + j];
      }
    }
  } else {  // W = Y^T: column j of the slice is Y[c0 + j, 0 .. N)
    if (yvec) {
      const int per = N / V;
      for (int e = tid; e < ncols * per; e += kResThreads) {
        const int j = e / per, i = (e - j * per) * V;
        const uint4 v = __ldg(reinterpret_cast<const uint4 *>(y + static_cast<size_t>(c0 + j) * N + i));
        const T *t = reinterpret_cast<const T *>(&v);
#pragma unroll
        for (int k = 0; k < V; ++k) w[(i + k) * ld + j] = t[k];
      }
    } else {
      for (int e = tid; e < ncols * N; e += kResThreads) {
        const int j = e / N, i = e - j * N;
        w[i * ld + j] = y[static_cast<size_t>(c0 + j) * N + i];
      }
    }
  }
  __syncthreads();

  // 2. sum of squares in W-row-major order (thread t: elements t, t + 256, ...
  //    of the slice, then a fixed tree) and the non-zero extent
  {
    float acc = 0.f;
    int rmax = -1, cmax = -1;
    for (int e = tid; e < m * ncols; e += kResThreads) {
      const int i = e / ncols, j = e - i * ncols;
      const float v = Elem<DT>::to_f(w[i * ld + j]);
      acc = fmaf(v, v, acc);
      if (v != 0.f) {
        rmax = max(rmax, i);
        cmax = max(cmax, j);
      }
    }
    acc = warp_sum(acc);
    rmax = warp_max(rmax);
    cmax = warp_max(cmax);
    if (lane == 0) {
      s_wsum[warp] = acc;
      s_wr[warp] = rmax;
      s_wc[warp] = cmax;
    }
    __syncthreads();
    if (tid == 0) {
      float t = 0.f;
      int rr = -1, cc = -1;
      for (int k = 0; k < kResThreads / 32; ++k) {
        t += s_wsum[k];
        rr = max(rr, s_wr[k]);
        cc = max(cc, s_wc[k]);
      }
      s_sum = t;
      s_rows = rr + 1;
      s_nse = cc + 1;
    }
  }
  res_sync(C);  // every CTA's sum and row extent are published
  if (tid == 0) {
    const float t = cluster_sum<C>(&s_sum);  // rank order
    int rv[C];
#pragma unroll
    for (int c = 0; c < C; ++c) rv[c] = C > 1 ? ld_cluster_i32(&s_rows, c) : s_rows;
    int rows = 0;
#pragma unroll
    for (int c = 0; c < C; ++c) rows = max(rows, rv[c]);
    s_r = 1.0f / (sqrtf(t) + p.eps);  // 1 / (||Y||_F + eps)
    s_meff = rows;
  }
  __syncthreads();
  const float r = s_r;
  const int meff = s_meff, nse = s_nse;

  // 3. the steps (meff is the same in every CTA of the cluster, so every CTA
  //    takes the same barriers)
  const int mb = (meff + 3) / 4;                  // 4-row blocks holding non-zero rows
  const int nblk = mb * (mb + 1) / 2;             // upper-triangle blocks
  const int kv = (nse + 7) / 8;                   // 8-column groups of the local contraction
  const int S = nblk > 0 ? max(1, min(kResThreads / nblk, kv)) : 1;
  const int kper = (kv + S - 1) / S;
  const int panel = 4 * (kResThreads / max(mb, 1));  // apply: columns per panel
  for (int step = 0; step < p.steps && meff > 0; ++step) {
    const float *co = p.coef[p.ncoef == 1 ? 0 : step];
    const float ca = co[0], cb = co[1], cc = co[2];
    const float gs = step == 0 ? r * r : 1.f, as0 = step == 0 ? r : 1.f;
    const float as = step == p.steps - 1 ? as0 * p.out_scale : as0;  // the last step applies the output scale
    float *Rs = R + (step & 1) * C * nent;  // this step's receive slots
    // ---- gram: partial 4 x 4 blocks of W_c W_c^T over k-slices of this CTA's columns
    if (tid < nblk * S) {
      const int b = tid / S, sl = tid - b * S;
      int bi, bj;
      upper_block(b, mb, bi, bj);
      const int g0 = sl * kper, g1 = min(kv, g0 + kper);
      float c4[4][4] = {};
      for (int g = g0; g < g1; ++g) {
        float xa[4][8], xb[4][8];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          ld8(w + (4 * bi + u) * ld + 8 * g, xa[u]);
          ld8(w + (4 * bj + u) * ld + 8 * g, xb[u]);
        }
#pragma unroll
        for (int k = 0; k < 8; ++k)
#pragma unroll
          for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int v = 0; v < 4; ++v) c4[u][v] = fmaf(xa[u][k], xb[v][k], c4[u][v]);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int v = 0; v < 4; ++v) part[(sl * nblk + b) * 16 + u * 4 + v] = c4[u][v];
    }
    __syncthreads();
    // slices in order -> this CTA's partial, stored into this rank's slot of
    // every CTA of the cluster (remote stores: nothing waits on them)
    for (int e = tid; e < nblk * 16; e += kResThreads) {
      const int b = e >> 4, u = (e >> 2) & 3, v = e & 3;
      float sum = 0.f;
      for (int sl = 0; sl < S; ++sl) sum += part[(sl * nblk + b) * 16 + u * 4 + v];
      float *slot = Rs + rank * nent + e;
      if (C > 1) {
#pragma unroll
        for (int c = 0; c < C; ++c) st_cluster_f32(slot, c, sum);
      } else {
        *slot = sum;
      }
    }
    res_sync(C);  // every CTA's partial has landed in every CTA
    // ---- A = gs * (sum of the partials in rank order), both triangles, from
    //      this CTA's own receive slots
    for (int e = tid; e < nblk * 16; e += kResThreads) {
      const int b = e >> 4, u = (e >> 2) & 3, w4 = e & 3;
      int bi, bj;
      upper_block(b, mb, bi, bj);
      if (bi < bj || u <= w4) {
        float sum = 0.f;
#pragma unroll
        for (int c = 0; c < C; ++c) sum += Rs[c * nent + e];
        sum *= gs;
        const int i = 4 * bi + u, j = 4 * bj + w4;
        A[i * ap + j] = sum;
        A[j * ap + i] = sum;
      }
    }
    __syncthreads();
    // ---- square: B = b A + c A A on upper blocks (symmetric, so both
    //      triangles); (A A)[i, j] = sum_k A[i, k] A[j, k], rows read 4 k at a time
    for (int b = tid; b < nblk; b += kResThreads) {
      int bi, bj;
      upper_block(b, mb, bi, bj);
      float c4[4][4] = {};
      for (int k = 0; k < 4 * mb; k += 4) {
        float ar[4][4];  // A[4 bi + u, k .. k + 3]: the warp's lanes share bi (broadcast)
#pragma unroll
        for (int u = 0; u < 4; ++u) ld4(A + (4 * bi + u) * ap + k, ar[u]);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          float ac[4];   // A[k + kk, 4 bj .. 4 bj + 3] = A[4 bj + v, k + kk]: contiguous across lanes
          ld4(A + (k + kk) * ap + 4 * bj, ac);
#pragma unroll
          for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int v = 0; v < 4; ++v) c4[u][v] = fmaf(ar[u][kk], ac[v], c4[u][v]);
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const int i = 4 * bi + u, j = 4 * bj + v;
          const float val = cb * A[i * ap + j] + cc * c4[u][v];
          B[i * ap + j] = val;
          B[j * ap + i] = val;
        }
    }
    __syncthreads();
    // ---- apply: W_c' = as (a W_c + B W_c), one column panel at a time
    for (int pc = 0; pc < nse; pc += panel) {
      const int rb = tid % mb, cbk = tid / mb;
      const int j0 = pc + 4 * cbk;
      const bool active = tid < mb * (panel / 4) && j0 < nse;
      float o4[4][4] = {};
      if (active) {
        for (int k = 0; k < 4 * mb; ++k) {
          float br[4], xr[4];
          ld4(B + k * ap + 4 * rb, br);  // B[k, 4 rb + u] = B[4 rb + u, k]: contiguous across lanes
          ld4(w + k * ld + j0, xr);      // the lanes of one column block share it (broadcast)
#pragma unroll
          for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int v = 0; v < 4; ++v) o4[u][v] = fmaf(br[u], xr[v], o4[u][v]);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          float xo[4];
          ld4(w + (4 * rb + u) * ld + j0, xo);
#pragma unroll
          for (int v = 0; v < 4; ++v) o4[u][v] = as * (ca * xo[v] + o4[u][v]);
        }
      }
      __syncthreads();  // every read of this panel happened
      if (active) {
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
          for (int v = 0; v < 4; ++v) w[(4 * rb + u) * ld + j0 + v] = Elem<DT>::from_f(o4[u][v]);
      }
      __syncthreads();
    }
  }
  if (p.steps == 0) {  // normalisation only
    const float rs = r * p.out_scale;
    for (int e = tid; e < meff * ld; e += kResThreads) w[e] = Elem<DT>::from_f(Elem<DT>::to_f(w[e]) * rs);
  }
  res_sync(C);  // no CTA leaves while another may still read its shared memory
  __syncthreads();

  // 4. write back the non-zero block (rows < meff, columns < nse, widened to
  //    16-byte words: the extra elements are the input's own zeros)
  const size_t ybytes = static_cast<size_t>(M) * N * sizeof(T);
  if (!tr) {
    if (yvec) {
      const int per = (nse + V - 1) / V;
      for (int e = tid; e < meff * per; e += kResThreads) {
        const int i = e / per, j = (e - i * per) * V;
        T *dst = y + static_cast<size_t>(i) * N + c0 + j;
        if (in_bounds(dst, 16, y, ybytes, p.status)) *reinterpret_cast<uint4 *>(dst) = *reinterpret_cast<const uint4 *>(w + i * ld + j);
      }
    } else {
      for (int e = tid; e < meff * nse; e += kResThreads) {
        const int i = e / nse, j = e - i * nse;
        T *dst = y + static_cast<size_t>(i) * N + c0 + j;
        if (in_bounds(dst, sizeof(T), y, ybytes, p.status)) *dst = w[i * ld + j];
      }
    }
  } else {
    if (yvec) {
      const int per = (meff + V - 1) / V;
      for (int e = tid; e < nse * per; e += kResThreads) {
        const int j = e / per, i = (e - j * per) * V;
        uint4 v;
        T *t = reinterpret_cast<T *>(&v);
#pragma unroll
        for (int k = 0; k < V; ++k) t[k] = w[(i + k) * ld + j];
        T *dst = y + static_cast<size_t>(c0 + j) * N + i;
        if (in_bounds(dst, 16, y, ybytes, p.status)) *reinterpret_cast<uint4 *>(dst) = v;
      }
    } else {
      for (int e = tid; e < nse * meff; e += kResThreads) {
        const int j = e / meff, i = e - j * meff;
        T *dst = y + static_cast<size_t>(c0 + j) * N + i;
        if (in_bounds(dst, sizeof(T), y, ybytes, p.status)) *dst = w[i * ld + j];
      }
    }
  }
}

template <int DT, int C>
int launch_resident_t(const ResParams &p, int smem, cudaStream_t s) {
  auto k = ns_resident_kernel<DT, C>;
  static SmemOptIn opt_in;
  if (opt_in.ensure(reinterpret_cast<const void *>(k), smem)) return -1;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(p.nmats * C, 1, 1);
  cfg.blockDim = dim3(kResThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, k, p) != cudaSuccess) {
    cudaGetLastError();
    return -1;
  }
  count_launch();
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

template <int DT>
int launch_resident_dt(const ResParams &p, int smem, cudaStream_t s) {
  switch (p.cluster) {
    case 1: return launch_resident_t<DT, 1>(p, smem, s);
    case 2: return launch_resident_t<DT, 2>(p, smem, s);
    case 4: return launch_resident_t<DT, 4>(p, smem, s);
    case 8: return launch_resident_t<DT, 8>(p, smem, s);
    default: return -1;
  }
}

}  // namespace

int launch_resident(const ResParams &p, int smem, cudaStream_t s) {
  if (p.nmats <= 0) return 0;
  if (p.dtype == kBF16) return launch_resident_dt<kBF16>(p, smem, s);
  return launch_resident_dt<kF32>(p, smem, s);
}

}  // namespace ns
