// ns_simt.cu -- CUDA-core kernels of libns:
//   * per-matrix Frobenius norm (partial sums) and non-zero extent (fp32 path),
//   * the per-matrix scale from the bf16 norm pass's tile sums,
//   * preparation: normalise by ||Y||_F + eps, round to the working type and
//     write both orientations W and W^T,
//   * the fp32 path's preparation for the tensor cores (three bf16 slices),
//   * the fp32 tiled CUDA-core GEMM phases (gram / square / apply), used for
//     large fp32 matrices under ns_set_f32_gemm(NS_F32_SIMT).
// The bf16 norm pass lives in ns_norm.cu, the bf16 tensor-core phases in
// ns_tc.cu, the shared-memory resident kernel for small matrices in
// ns_resident.cu.
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
  const float inv = p.to_user ? s_denom * p.out_scale : s_denom;
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
    const size_t dst_bytes = static_cast<size_t>(rows) * pitch * sizeof(T);  // the destination buffer
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
        if (in_bounds(out, 16, dst, dst_bytes, p.status)) *reinterpret_cast<uint4 *>(out) = w;
      } else {
        for (int u = 0; u < V && C + u < cols; ++u)
          if (in_bounds(out + u, sizeof(T), dst, dst_bytes, p.status))
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

// fp32 tensor-core path: one block per 64x64 tile of the caller's Y (tiles
// located as in ns_prep_kernel). Writes w = y / (||Y||_F + eps), computed in
// fp32, as its three bf16 slices h = bf16(w), m = bf16(w - h),
// l = bf16(w - h - m) into the three slices of the first iterate buffer s[0]
// (the caller's orientation, row pitch ps, slices M * ps elements apart).
// Each thread moves runs of 8 elements: two 16-byte loads of Y when its rows
// are 16-byte aligned, one 16-byte store per slice.
__global__ void __launch_bounds__(256) ns_split_prep_kernel(PrepParams p) {
  const int bid = blockIdx.x;
  int lo = 0, hi = p.nmats;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (p.tile_prefix[mid] <= bid) lo = mid; else hi = mid;
  }
  const int mat = lo;
  const MatDesc &d = p.mats[mat];
  const int M = d.M, N = d.N, ps = d.ps;
  const int local = bid - p.tile_prefix[mat];
  const int tcols = (N + kPrepTile - 1) / kPrepTile;
  const int r0 = (local / tcols) * kPrepTile, c0 = (local % tcols) * kPrepTile;
  const float *y = static_cast<const float *>(d.user);
  const bool vec = (N % 4 == 0) && ((reinterpret_cast<uintptr_t>(y) & 15) == 0);
  __nv_bfloat16 *s0 = static_cast<__nv_bfloat16 *>(d.s[0]);
  const size_t slice = static_cast<size_t>(M) * ps;

  __shared__ float s_denom;
  const int tid = threadIdx.x;
  if (tid < 32) {
    float v = 0.f;
    for (int i = tid; i < kNormBlocks; i += 32) v += p.partials[mat * kNormBlocks + i];
    v = warp_sum(v);
    if (tid == 0) s_denom = 1.0f / (sqrtf(v) + p.eps);  // 1 / (||Y||_F + eps)
  }
  __syncthreads();
  const float inv = s_denom;
  constexpr int kRuns = kPrepTile * kPrepTile / 8 / 256;  // runs of 8 per thread
#pragma unroll
  for (int k = 0; k < kRuns; ++k) {
    const int q = tid + k * 256, rr = q / (kPrepTile / 8), cg = q % (kPrepTile / 8);
    const int r = r0 + rr, c = c0 + cg * 8;
    if (r >= M || c >= N) continue;
    const float *src = y + static_cast<size_t>(r) * N + c;
    const int n = min(8, N - c);
    float w[8];
    if (vec && n == 8) {
      const float4 a = __ldg(reinterpret_cast<const float4 *>(src));
      const float4 b = __ldg(reinterpret_cast<const float4 *>(src) + 1);
      w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
      w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
    } else {
#pragma unroll
      for (int u = 0; u < 8; ++u) w[u] = u < n ? src[u] : 0.f;
    }
    uint32_t bits[3][8];  // the slices' bf16 bit patterns
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      float v = w[u] * inv;
#pragma unroll
      for (int z = 0; z < 3; ++z) {
        const __nv_bfloat16 h = __float2bfloat16_rn(v);
        bits[z][u] = __bfloat16_as_ushort(h);
        v -= __bfloat162float(h);  // exact
      }
    }
#pragma unroll
    for (int z = 0; z < 3; ++z) {
      __nv_bfloat16 *base = s0 + z * slice;
      __nv_bfloat16 *dst = base + static_cast<size_t>(r) * ps + c;  // 16-byte aligned: ps and c are multiples of 8
      if (n == 8) {
        const uint4 o = make_uint4(bits[z][0] | (bits[z][1] << 16), bits[z][2] | (bits[z][3] << 16),
                                   bits[z][4] | (bits[z][5] << 16), bits[z][6] | (bits[z][7] << 16));
        if (in_bounds(dst, 16, base, slice * 2, p.status)) *reinterpret_cast<uint4 *>(dst) = o;
      } else {
        for (int u = 0; u < n; ++u)
          if (in_bounds(dst + u, 2, base, slice * 2, p.status))
            dst[u] = __ushort_as_bfloat16(static_cast<unsigned short>(bits[z][u]));
      }
    }
  }
}

int launch_split_prep(const PrepParams &p, int total_tiles, cudaStream_t s) {
  if (total_tiles <= 0) return 0;
  ns_split_prep_kernel<<<total_tiles, 256, 0, s>>>(p);
  count_launch();
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

// One block per matrix: the tile partial sums of the matrix in a fixed order
// (strided per thread, then a fixed tree) give r = 1 / (||Y||_F + eps), and
// the largest of the tiles' extents gives the matrix's non-zero extent.
__global__ void __launch_bounds__(256) ns_norm_finish_kernel(PrepParams p) {
  const int mat = blockIdx.x;
  const int t0 = p.tile_prefix[mat], t1 = p.tile_prefix[mat + 1];
  float v = 0.f;
  int er = 0, ec = 0;
  for (int i = t0 + static_cast<int>(threadIdx.x); i < t1; i += 256) {
    v += p.tile_partials[i];
    const int2 e = reinterpret_cast<const int2 *>(p.tile_ext)[i];
    er = max(er, e.x);
    ec = max(ec, e.y);
  }
  __shared__ float s_sum[8];
  __shared__ int s_r[8], s_c[8];
  v = warp_sum(v);
  er = warp_max(er);
  ec = warp_max(ec);
  if ((threadIdx.x & 31) == 0) {
    s_sum[threadIdx.x >> 5] = v;
    s_r[threadIdx.x >> 5] = er;
    s_c[threadIdx.x >> 5] = ec;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    int rr = 0, cc = 0;
    for (int w = 0; w < 8; ++w) {
      t += s_sum[w];
      rr = max(rr, s_r[w]);
      cc = max(cc, s_c[w]);
    }
    p.rscale[mat] = 1.0f / (sqrtf(t) + p.eps);
    p.ext[2 * mat + 0] = rr;
    p.ext[2 * mat + 1] = cc;
  }
}

int launch_norm_finish(const PrepParams &p, cudaStream_t s) {
  if (p.nmats <= 0) return 0;
  ns_norm_finish_kernel<<<p.nmats, 256, 0, s>>>(p);
  count_launch();
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
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
          const size_t bytes = static_cast<size_t>(m) * pm * 4;
          if (PHASE == 1) out = p.cb * static_cast<const float *>(d.a)[static_cast<size_t>(r) * pm + c] + p.cc * val;
          float *d0 = dst + static_cast<size_t>(r) * pm + c, *d1 = dst + static_cast<size_t>(c) * pm + r;
          if (in_bounds(d0, 4, dst, bytes, p.status)) *d0 = out;
          if (in_bounds(d1, 4, dst, bytes, p.status)) *d1 = out;
        }
      } else {
        if (r < n && c < m) {
          const float *xt = static_cast<const float *>(d.xt[cur]);
          const float out0 = p.ca * xt[static_cast<size_t>(r) * pm + c] + val;
          const float out = p.final_step ? out0 * p.out_scale : out0;
          if (!p.final_step) {
            float *xt1 = static_cast<float *>(d.xt[cur ^ 1]), *x = static_cast<float *>(d.x);
            float *d0 = xt1 + static_cast<size_t>(r) * pm + c, *d1 = x + static_cast<size_t>(c) * pn + r;
            if (in_bounds(d0, 4, xt1, static_cast<size_t>(n) * pm * 4, p.status)) *d0 = out;
            if (in_bounds(d1, 4, x, static_cast<size_t>(m) * pn * 4, p.status)) *d1 = out;
          } else {
            float *u = static_cast<float *>(d.user);
            float *d0 = d.transposed ? u + static_cast<size_t>(r) * d.N + c : u + static_cast<size_t>(c) * d.N + r;
            if (in_bounds(d0, 4, u, static_cast<size_t>(d.M) * d.N * 4, p.status)) *d0 = out;
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
