// ns_norm.cu -- the norm pass of the bf16 path: the one read of every caller
// matrix Y before the first step.
//
// For each matrix it produces the sum of squares of every 64 x 64 tile of W
// (W = Y, or Y^T when M > N) and the last non-zero row and column of every
// tile of Y (the finish kernel reduces both per matrix, without atomics), and,
// when the first step cannot read Y itself through TMA, an exact copy of Y in
// the first iterate buffer. The scale 1/(||Y||_F + eps) is formed from the
// tile sums by ns_norm_finish_kernel and applied inside the first step's GEMM
// epilogues (A = r^2 Y Y^T, W_1 = r (a Y + B Y)), so Y is read once here and
// the first normalised iterate is never rounded.
//
// Every sum is taken in W's orientation: an 8 x 8 sub-block in W-row-major
// order, the 64 sub-block sums of a tile by a fixed tree over their W index,
// the tiles in W's tile order (ns_norm_finish_kernel). A matrix and its
// transpose therefore get bit-identical scales. The squares are exact in fp32
// (a bf16 has 8 significant bits); a sub-block sum is two fixed chains of
// fp32 fused multiply-adds (see subblock_sumsq).
//
// Work split: one warp per 64 x 64 tile of Y at a time (tiles strided over
// all warps of a persistent grid of two 256-thread blocks per SM). A tile is
// read as two halves of 32 rows; lane l holds the 8 x 8 sub-block
// (l / 8 + 4 h, l % 8) of half h as eight 16-byte rows (each copy instruction
// of the warp reads 4 rows x 128 contiguous bytes). Each lane streams its own
// rows into its own slots of a three-half-tile ring in shared memory with
// cp.async (16-byte copies that zero-fill past the matrix), two half-tiles
// ahead of the one it reduces, so the bytes in flight do not occupy
// registers: 16 warps per SM keep 128 KB in flight. A lane reads back only
// what it copied itself, so the ring needs no barrier. Rows that are not
// 16-byte aligned (N not a multiple of 8, or an unaligned Y) are loaded
// element by element into the same slots instead. Zero extents are tested a
// 16-byte word at a time: a row is non-zero when the OR of its words has a
// non-zero magnitude bit, a column when the OR over the rows has one in that
// column's half-word; a lane's last row and last column are tested first.
#include <cuda_runtime.h>

#include <algorithm>

#include "ns_device.cuh"

namespace ns {

namespace {

constexpr uint32_t kMagnitude = 0x7FFF7FFFu;  // both halves' bits except the signs (-0 counts as zero)

// Where tile `tile` of the call's concatenated tile lists lies.
struct TileLoc {
  const __nv_bfloat16 *y;  // the caller's matrix
  __nv_bfloat16 *copy;     // first iterate buffer to copy Y into, or null (step 1 reads Y itself)
  int mat, M, N;
  int r0, c0;
  int wtile;               // the tile's index in W's tile grid, offset by the matrix's first tile
  int tr;                  // W = Y^T
  int vec;                 // rows of Y are 16-byte aligned: one 16-byte load per 8 elements
};

// q = n / d, r = n % d for 0 <= n, 0 < d: an fp32 estimate corrected by one
// step (the estimate is within one of q when n < 2^20), else a division.
__device__ __forceinline__ void divmod(int n, int d, int &q, int &r) {
  if (n < (1 << 20)) {
    q = __float2int_rz(__fdividef(static_cast<float>(n), static_cast<float>(d)));
    r = n - q * d;
    if (r < 0) {
      --q;
      r += d;
    } else if (r >= d) {
      ++q;
      r -= d;
    }
  } else {
    q = n / d;
    r = n - q * d;
  }
}

// The matrix a warp is in, kept while its tiles (visited in increasing
// order) stay in that matrix: a tile's location then needs no memory access,
// and a new matrix's record is read once, when the warp crosses into it.
struct Locator {
  int mat, base, end;  // the matrix and its tiles [base, end) in the call's tile numbering
  const __nv_bfloat16 *y;
  __nv_bfloat16 *copy;
  int M, N, tr, vec, tcols, mtiles;
};

__device__ __forceinline__ void locator_load(const PrepParams &p, Locator &L) {
  const MatDesc &d = p.mats[L.mat];
  L.end = p.tile_prefix[L.mat + 1];
  L.M = d.M;
  L.N = d.N;
  L.tr = d.transposed;
  L.y = static_cast<const __nv_bfloat16 *>(d.user);
  L.copy = d.direct ? nullptr : static_cast<__nv_bfloat16 *>(d.s[0]);
  L.vec = (L.N % 8 == 0) && ((reinterpret_cast<uintptr_t>(L.y) & 15) == 0);
  L.tcols = (L.N + kPrepTile - 1) / kPrepTile;
  L.mtiles = (L.M + kPrepTile - 1) / kPrepTile;
}

// The warp's first tile: a binary search over the tile prefix counts.
__device__ __forceinline__ void locator_start(const PrepParams &p, int tile, Locator &L) {
  int lo = 0, hi = p.nmats;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (p.tile_prefix[mid] <= tile) lo = mid; else hi = mid;
  }
  L.mat = lo;
  L.base = p.tile_prefix[lo];
  locator_load(p, L);
}

// A later tile of the same warp (tile >= every tile located before).
__device__ __forceinline__ TileLoc locate(const PrepParams &p, int tile, Locator &L) {
  while (tile >= L.end) {
    ++L.mat;
    L.base = L.end;
    locator_load(p, L);
  }
  TileLoc t;
  t.mat = L.mat;
  t.M = L.M;
  t.N = L.N;
  t.tr = L.tr;
  t.y = L.y;
  t.copy = L.copy;
  t.vec = L.vec;
  const int local = tile - L.base;
  int tr_, tc_;
  divmod(local, L.tcols, tr_, tc_);
  t.r0 = tr_ * kPrepTile;
  t.c0 = tc_ * kPrepTile;
  t.wtile = L.base + (t.tr ? tc_ * L.mtiles + tr_ : local);
  return t;
}

constexpr int kRing = 3;                         // half-tiles per lane in flight or being reduced
constexpr int kSlotBytes = 8 * 16;               // one lane's rows of one half-tile
constexpr int kSlot = 32 * kSlotBytes;          // one half-tile of the warp (4 KB)
constexpr int kWarpRingBytes = kRing * kSlot;
constexpr int kNormSmem = 8 * kWarpRingBytes;    // 96 KB per 256-thread block

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Start this lane's copies of its 8 rows of 8 columns in half h of the tile
// into its slot (row r at slot + r * 16 * 32: lanes interleaved, so the later
// 16-byte shared-memory reads of a warp are contiguous).
__device__ __forceinline__ void issue_half(const TileLoc &t, int h, int lane, uint8_t *slot) {
  const int C = t.c0 + (lane & 7) * 8;
  const int R0 = t.r0 + ((lane >> 3) + 4 * h) * 8;
  if (t.vec) {
    // rows are whole 16-byte words; rows past the matrix are zero-filled
    const uint32_t dst = smem_u32(slot);
    const bool col_in = C < t.N;
    const __nv_bfloat16 *src = t.y + (col_in ? static_cast<size_t>(R0) * t.N + C : 0);
    const size_t pitch = col_in ? static_cast<size_t>(t.N) : 0;
    const int rows_in = col_in ? min(8, t.M - R0) : 0;
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const bool in = r < rows_in;
      cp_async16(dst + r * 16 * 32, in ? src : t.y, in ? 16u : 0u);
      src += pitch;
    }
  } else {
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const int R = R0 + r;
      uint4 w = make_uint4(0, 0, 0, 0);
      if (R < t.M && C < t.N) {
        const __nv_bfloat16 *src = t.y + static_cast<size_t>(R) * t.N + C;
        uint32_t e[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) e[k] = C + k < t.N ? static_cast<uint32_t>(__bfloat16_as_ushort(src[k])) : 0u;
        w = make_uint4(e[0] | (e[1] << 16), e[2] | (e[3] << 16), e[4] | (e[5] << 16), e[6] | (e[7] << 16));
      }
      *reinterpret_cast<uint4 *>(slot + r * 16 * 32) = w;
    }
  }
}

__device__ __forceinline__ void read_half(const uint8_t *slot, uint4 (&v)[8]) {
#pragma unroll
  for (int r = 0; r < 8; ++r) v[r] = *reinterpret_cast<const uint4 *>(slot + r * 16 * 32);
}

__device__ __forceinline__ uint32_t word(const uint4 &v, int q) { return q == 0 ? v.x : q == 1 ? v.y : q == 2 ? v.z : v.w; }
// fp32 value of the low / high bf16 of a word (exact)
__device__ __forceinline__ float lo_f(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi_f(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Sum of squares of the lane's sub-block in W's orientation: four chains of
// fused multiply-adds, one per parity of W's row and of W's column, each in
// W-row-major order (one paired fp32 FMA advances the even- and odd-column
// chains of a row), then (even row: even + odd column) + (odd row: even +
// odd column). For W = Y a 16-byte row of Y holds a W row's two chains side
// by side; for W = Y^T, W(i, 2q) and W(i, 2q + 1) are Y(2q, i) and
// Y(2q + 1, i), the same half of the same word in two adjacent rows.
__device__ __forceinline__ float subblock_sumsq(const uint4 (&v)[8], int tr) {
  float2 acc[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
  if (!tr) {
#pragma unroll
    for (int wi = 0; wi < 8; ++wi)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t w = word(v[wi], q);
        const float2 x = make_float2(lo_f(w), hi_f(w));
        acc[wi & 1] = __ffma2_rn(x, x, acc[wi & 1]);
      }
  } else {
#pragma unroll
    for (int wi = 0; wi < 8; ++wi)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t e = word(v[2 * q], wi >> 1), o = word(v[2 * q + 1], wi >> 1);
        const float2 x = (wi & 1) ? make_float2(hi_f(e), hi_f(o)) : make_float2(lo_f(e), lo_f(o));
        acc[wi & 1] = __ffma2_rn(x, x, acc[wi & 1]);
      }
  }
  return (acc[0].x + acc[0].y) + (acc[1].x + acc[1].y);
}

// Reduce half h of a tile held in v: the sub-block sum into the warp's slot
// table (by W index), the lane's extents, and the copy when there is one.
__device__ __forceinline__ void reduce_half(const TileLoc &t, int h, int lane, const uint4 (&v)[8], float *slots,
                                            int &ext_r, int &ext_c, int *status) {
  const int br = (lane >> 3) + 4 * h, bc = lane & 7;
  const int R0 = t.r0 + br * 8, C = t.c0 + bc * 8;
  // extents: the last of the 8 rows, and the last of the 8 columns, that
  // holds a non-zero. Dense data has both in the lane's last row and column,
  // which are tested first; the full scans run only when one of them is zero.
  if ((v[7].x | v[7].y | v[7].z | v[7].w) & kMagnitude) {
    ext_r = max(ext_r, R0 + 7);
  } else {
    uint32_t rows = 0;
#pragma unroll
    for (int r = 0; r < 7; ++r) rows |= (((v[r].x | v[r].y | v[r].z | v[r].w) & kMagnitude) != 0 ? 1u : 0u) << r;
    if (rows) ext_r = max(ext_r, R0 + 31 - __clz(rows));
  }
  const uint32_t last_col = v[0].w | v[1].w | v[2].w | v[3].w | v[4].w | v[5].w | v[6].w | v[7].w;
  if (last_col & 0x7FFF0000u) {
    ext_c = max(ext_c, C + 7);
  } else {
    uint4 cols = make_uint4(0, 0, 0, last_col);
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      cols.x |= v[r].x;
      cols.y |= v[r].y;
      cols.z |= v[r].z;
    }
    const uint32_t cmask = ((cols.x & 0x7FFFu) ? 1u : 0u) | ((cols.x & 0x7FFF0000u) ? 2u : 0u) |
                           ((cols.y & 0x7FFFu) ? 4u : 0u) | ((cols.y & 0x7FFF0000u) ? 8u : 0u) |
                           ((cols.z & 0x7FFFu) ? 16u : 0u) | ((cols.z & 0x7FFF0000u) ? 32u : 0u) |
                           ((cols.w & 0x7FFFu) ? 64u : 0u);
    if (cmask) ext_c = max(ext_c, C + 31 - __clz(cmask));
  }
  // exact copy into the first iterate buffer (its pitch: N rounded up to 8 elements)
  if (t.copy && C < t.N) {
    const int ps = (t.N + 7) & ~7;
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      __nv_bfloat16 *dst = t.copy + static_cast<size_t>(R0 + r) * ps + C;
      if (R0 + r < t.M && in_bounds(dst, 16, t.copy, static_cast<size_t>(t.M) * ps * 2, status))
        *reinterpret_cast<uint4 *>(dst) = v[r];
    }
  }
  slots[t.tr ? bc * 8 + br : br * 8 + bc] = subblock_sumsq(v, t.tr);
}


__global__ void __launch_bounds__(256, 2) ns_norm_tiles_kernel(PrepParams p, int total_tiles) {
  extern __shared__ __align__(16) uint8_t norm_smem[];
  __shared__ float s_blk[8][64];  // per warp: sub-block sums of its tile, by W index
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = gridDim.x * 8;
  float *slots = s_blk[warp];
  uint8_t *ring = norm_smem + warp * kWarpRingBytes + lane * 16;
  int tile = blockIdx.x * 8 + warp;
  if (tile >= total_tiles) return;  // whole warps only; no block-wide barrier follows
  // The copies run two half-tiles (one tile) ahead of the reduction: while
  // the halves of `tile` are reduced, the halves of `next` are being copied.
  // Every half commits one copy group (empty past the end), so waiting until
  // at most kRing - 1 groups are pending means the half about to be reduced
  // has landed.
  Locator L;
  locator_start(p, tile, L);
  TileLoc loc = locate(p, tile, L);
  issue_half(loc, 0, lane, ring);
  cp_async_commit();
  issue_half(loc, 1, lane, ring + kSlot);
  cp_async_commit();
  int next = tile + nwarps;
  TileLoc nloc = loc;
  if (next < total_tiles) nloc = locate(p, next, L);
  int in_slot = 2, out_slot = 0;
  for (;;) {
    int ext_r = -1, ext_c = -1;  // this tile's last non-zero row and column (caller's orientation)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      if (next < total_tiles) issue_half(nloc, h, lane, ring + in_slot * kSlot);
      cp_async_commit();
      in_slot = in_slot + 1 == kRing ? 0 : in_slot + 1;
      cp_async_wait<kRing - 1>();  // this lane's copies of half h of `tile` have landed
      uint4 v[8];
      read_half(ring + out_slot * kSlot, v);
      out_slot = out_slot + 1 == kRing ? 0 : out_slot + 1;
      reduce_half(loc, h, lane, v, slots, ext_r, ext_c, p.status);
    }
    __syncwarp();
    float s = slots[2 * lane] + slots[2 * lane + 1];
    s = warp_sum(s);  // xor butterfly: every lane ends with the same value
    ext_r = warp_max(ext_r);
    ext_c = warp_max(ext_c);
    if (lane == 0) {
      p.tile_partials[loc.wtile] = s;
      // the tile's extents, one past the last non-zero row / column (0: none),
      // at the tile's place in the caller's tile order; ns_norm_finish_kernel
      // takes the maximum per matrix (no atomics)
      reinterpret_cast<int2 *>(p.tile_ext)[tile] = make_int2(ext_r + 1, ext_c + 1);
    }
    __syncwarp();
    if (next >= total_tiles) break;
    tile = next;
    loc = nloc;
    next += nwarps;
    if (next < total_tiles) nloc = locate(p, next, L);
  }
  cp_async_wait<0>();
}

}  // namespace

int launch_norm_tiles(const PrepParams &p, int total_tiles, int max_blocks, cudaStream_t s) {
  if (total_tiles <= 0) return 0;
  const int blocks = std::min((total_tiles + 7) / 8, std::max(max_blocks, 1));
  static SmemOptIn opt_in;
  if (opt_in.ensure(reinterpret_cast<const void *>(ns_norm_tiles_kernel), kNormSmem)) return -1;
  ns_norm_tiles_kernel<<<blocks, 256, kNormSmem, s>>>(p, total_tiles);
  count_launch();
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace ns
