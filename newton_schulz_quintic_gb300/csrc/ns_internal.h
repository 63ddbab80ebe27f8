// ns_internal.h -- structures shared by the host planner and the kernels of
// libns (batched quintic Newton-Schulz on sm_103a). Not part of the C ABI.
//
// Working layout of one matrix on the large-matrix path. The caller's matrix
// Y is M x N row-major. The iteration works on W (m x n, m = min(M,N)),
// W = Y^T when M > N ("transposed"). The workspace holds, per matrix:
//   x      W      m x n   row pitch pn = round_up(n, 8) elements
//   xt[2]  W^T    n x m   row pitch pm = round_up(m, 8); ping-pong across steps
//   a      A      m x m   row pitch pm  (A = W W^T, symmetric)
//   b      B      m x m   row pitch pm  (B = b A + c A^2, symmetric)
// All five are row-major with the contraction index contiguous for the way
// they are consumed, so every GEMM reads both operands K-major:
//   gram    A[i,j]  = sum_k x[i,k]  x[j,k]        (K = n)
//   square  C[i,j]  = sum_k a[i,k]  a[j,k]        (K = m; A symmetric so A A = A A^T)
//   apply   D[j,i]  = sum_k xt[j,k] b[i,k]        (K = m; D = (B W)^T)
// Pitches are multiples of 16 bytes so TMA can address every row.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace ns {

enum StoreType : int { kF32 = 0, kBF16 = 1 };

constexpr int kMaxTableSteps = 32;  // longest per-step coefficient table

// Tile of one GEMM phase: tile rows [row0, row0+BM), tile cols [col0, col0+BN)
// of matrix `mat` (index into the matrix descriptor table).
struct Tile {
  int mat;
  int row0;
  int col0;
  int pad;
};

struct MatDesc {  // CUtensorMap members keep it 64-byte aligned or more
  CUtensorMap tm_x;      // x,  box {64, 128}
  CUtensorMap tm_a;      // a,  box {64, 128}
  CUtensorMap tm_b;      // b,  box {64, 128}
  CUtensorMap tm_xt[2];  // xt, box {64, 128}
  void *x;
  void *a;
  void *b;
  void *xt[2];
  void *user;            // caller's Y (M x N row-major)
  int M, N;              // caller's shape
  int m, n;              // working shape
  int pm, pn;            // pitches (elements) of m-wide and n-wide buffers
  int transposed;        // 1 when M > N
  int index;             // position in the caller's batch
  int t01, t2;           // tensor-core path: pair tiles of this matrix per gram/square and per apply
};

// Small matrices done entirely in one CTA (shared-memory resident).
struct ResDesc {
  void *user;
  int M, N;
  int m, n;
  int transposed;
  int pad;
};

// Kernel parameters shared by the phase kernels.
struct PhaseParams {
  const Tile *tiles;
  int ntiles;
  const MatDesc *mats;
  const int *ext;        // per matrix: {rows_eff, cols_eff} in the caller's orientation
  int *status;           // device status word
  float ca, cb, cc;      // coefficients a, b, c
  int step;              // 0-based step (selects xt ping-pong buffer)
  int final_step;        // 1 on the last step: write the caller's matrix
};

// Parameters of the tensor-core GEMM kernel. Its work is the item sequence
// step-major, then phase (gram, square, apply), then the phase's tile list
// (all matrices, largest ns_cost first): item g of a step lies in
// [0, 2*n01 + n2). A launch runs items [g_begin, g_end) of that sequence.
// With wait != 0 an item first waits until every item of the same matrix in
// earlier phases is complete (per-matrix completion counters `done`), so one
// launch can run every step and phase; with wait == 0 the launches themselves
// order the phases.
struct TcParams {
  const Tile *tiles01;  // gram / square pair tiles
  const Tile *tiles2;   // apply pair tiles
  int n01, n2;
  int g_begin, g_end;
  int steps;            // total steps of the call (the last one writes the caller's matrices)
  int wait;
  const MatDesc *mats;
  const int *ext;       // per matrix {rows_eff, cols_eff} in the caller's orientation
  int *status;
  int *done;            // per matrix completion counter (zeroed by the host per call)
  int ncoef;            // 1: coef[0] for every step; else coef[step]
  float coef[kMaxTableSteps][3];
};

// Norm / preparation kernel parameters.
struct PrepParams {
  const MatDesc *mats;
  int nmats;
  float *partials;       // nmats * kNormBlocks partial sums of squares
  int *ext;              // nmats * 2
  const int *tile_prefix;  // nmats + 1 prefix counts of 64x64 tiles of Y
  float eps;
  int dtype;             // StoreType of the caller's data == workspace store type
  int to_user;           // 1: write the normalised matrix back to the caller (steps == 0)
};

struct ResParams {
  const ResDesc *mats;
  int nmats;
  int dtype;
  int steps;
  int ncoef;                        // 1: coef[0] for every step; else coef[step]
  float coef[kMaxTableSteps][3];    // (a, b, c)
  float eps;
};

constexpr int kNormBlocks = 128;  // partial-sum blocks per matrix
constexpr int kPrepTile = 64;     // Y tile edge of the preparation kernel

// tcgen05 GEMM tile (bf16 path). Tiles are processed by 2-CTA clusters: a
// tile list entry covers kTcPairM x kTcBN outputs, CTA rank r of the cluster
// computes rows [row0 + r*kTcBM, row0 + (r+1)*kTcBM) and the pair shares the
// kTcBN-row second operand through TMA multicast.
constexpr int kTcBM = 128;
constexpr int kTcBN = 256;
constexpr int kTcBK = 64;
constexpr int kTcCluster = 2;
constexpr int kTcPairM = kTcCluster * kTcBM;
// SIMT GEMM tile (fp32 path)
constexpr int kSimtBM = 64;
constexpr int kSimtBN = 64;

// host-side launchers (defined in the .cu files)
int launch_norm(const PrepParams &p, cudaStream_t s);
int launch_prep(const PrepParams &p, int total_tiles, cudaStream_t s);
int launch_resident(const ResParams &p, int maxm, int smem_bytes, cudaStream_t s);
int launch_simt_phase(int phase, const PhaseParams &p, cudaStream_t s);
int launch_tc(const TcParams &p, int max_ctas, cudaStream_t s);
int tc_smem_bytes();
int launch_wait_probe(int *status, uint64_t limit_ns, int *gave_up, cudaStream_t s);
int resident_smem_bytes(int m, int n, int dtype);

void count_launch();

}  // namespace ns
