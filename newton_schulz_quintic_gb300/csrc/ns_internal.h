// ns_internal.h -- structures shared by the host planner and the kernels of
// libns (batched quintic Newton-Schulz on sm_103a). Not part of the C ABI.
//
// Working layout of one matrix on the large-matrix paths. The caller's
// matrix Y is M x N row-major. The iteration works on W (m x n,
// m = min(M,N)), W = Y^T when M > N ("transposed").
//
// bf16 tensor-core path: every iterate is kept in the caller's orientation
// (Y-shaped, so W^T when transposed) and the GEMMs read whichever operand
// order that gives, K-major or MN-major (tcgen05 reads both):
//   s[2]   iterates  M x N   row pitch ps = round_up(N, 8); ping-pong across
//                            steps (step 0 reads Y itself when TMA can address it)
//   a      A         m x m   row pitch pm = round_up(m, 8)  (A = W W^T, symmetric;
//                            only its upper 256 x 256 tiles are stored, whole)
//   b      B         m x m   row pitch pm  (B = b A + c A^2, symmetric; upper tiles)
//   gram    A[i,j] = sum_k W[i,k] W[j,k]    (K = n; MN-major operands when transposed)
//   square  C[i,j] = sum_k A[i,k] A[j,k]    (K = m; A symmetric so A A = A A^T;
//                                            A[i,k] with k left of i's diagonal tile is
//                                            read MN-major as A[k,i] from an upper tile)
//   apply   not transposed: D = B W   (W read MN-major), D[i,j] over m x n
//           transposed:     D = W^T B (W^T = the iterate, K-major), D over n x m
//           either way D is the next iterate in the caller's orientation.
// fp32 tensor-core path: as the bf16 path, but every tensor (s[2], a, b) is
// three bf16 slices x = h + m + l (h = bf16(x), m = bf16(x - h),
// l = bf16(x - h - m)), stored as three consecutive buffers of the shape
// above; step 0 reads s[0], which the preparation fills with the slices of
// Y / (||Y||_F + eps), and the last step writes fp32 into the caller's Y.
// fp32 CUDA-core path (optional): both orientations are kept, all reads K-major:
//   x      W      m x n   row pitch pn = round_up(n, 8)
//   xt[2]  W^T    n x m   row pitch pm; ping-pong across steps
//   a, b   as above
// Pitches are multiples of 16 bytes so TMA can address every row.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace ns {

enum StoreType : int { kF32 = 0, kBF16 = 1 };

constexpr int kMaxTableSteps = 32;  // longest per-step coefficient table

// Default upper bound of any single bounded wait inside a kernel (passed to
// the kernels as a parameter). A correct kernel never gets near it; if it is
// reached the kernel records NS_ETIMEOUT and winds down.
constexpr uint64_t kWaitLimitNs = 4000000000ull;  // 4 s

// Tile of one GEMM phase: tile rows [row0, row0+BM), tile cols [col0, col0+BN)
// of matrix `mat` (index into the matrix descriptor table).
struct Tile {
  int mat;
  int row0;
  int col0;
  int pad;
};

struct MatDesc {  // CUtensorMap members keep it 64-byte aligned or more
  // bf16 path, 128-byte swizzle. K-major loads take one box of 64 columns x
  // 128 rows; MN-major loads two boxes of 64 x 64 (the swizzle span limits
  // a box row to 128 bytes, i.e. 64 elements of the MN index)
  CUtensorMap tm_a;       // a, box {64, 128}
  CUtensorMap tm_b;       // b, box {64, 128}
  CUtensorMap tm_a_mn;    // a, box {64, 64} (rows left of the diagonal, read from the mirrored upper tiles)
  CUtensorMap tm_b_mn;    // b, box {64, 64}
  CUtensorMap tm_s[2];    // s[0], s[1], box {64, 128}
  CUtensorMap tm_s_mn[2]; // s[0], s[1], box {64, 64}
  CUtensorMap tm_y;       // the caller's Y (used when `direct`), box {64, 128}
  CUtensorMap tm_y_mn;    // the caller's Y, box {64, 64}
  void *x;               // fp32 path: W
  void *xt[2];           // fp32 path: W^T ping-pong
  void *s[2];            // bf16 path: iterates in the caller's orientation
  void *a;
  void *b;
  void *user;            // caller's Y (M x N row-major)
  int M, N;              // caller's shape
  int m, n;              // working shape
  int pm, pn, ps;        // pitches (elements) of m-wide, n-wide and N-wide buffers
  int transposed;        // 1 when M > N
  int direct;            // bf16 path: step 0 reads Y itself (else an exact copy in s[0])
  int index;             // position in the caller's batch
  int t01, t2;           // tensor-core path: pair tiles of this matrix per gram/square and per apply
};

// Small matrices done entirely in shared memory, each by a cluster of CTAs
// that split W's columns into slices of `ns` columns.
struct ResDesc {
  void *user;
  int M, N;
  int m, n;
  int transposed;
  int ns;
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
  float out_scale;       // the last step's result is multiplied by it before the write
};

// Parameters of the tensor-core GEMM kernel. Its work is the item sequence
// step-major, then phase (gram, square, apply), then the phase's tile list
// (all matrices, largest ns_cost first): item g of a step lies in
// [0, 2*n01 + n2). A launch runs items [g_begin, g_end) of that sequence.
// With wait != 0 an item first waits until every item of the same matrix in
// earlier phases is complete (per-matrix completion counters `done`), so one
// launch can run every step and phase; with wait == 0 the launches themselves
// order the phases. With tickets != 0 the CTA pairs take items from the
// counter `ticket` (zeroed by the host per call) in sequence order, so the
// items in flight stay contiguous; otherwise pair c takes c, c + #pairs, ...
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
  int *ticket;          // next item to hand out, relative to g_begin (zeroed by the host per call)
  int tickets;          // 1: items by ticket; 0: static stride
  int split;            // 1: fp32 path, every tensor three bf16 slices (per-phase launches only)
  const float *rscale;  // per matrix 1 / (||Y||_F + eps): step 0 scales gram by its square and apply by it
  uint64_t wait_limit_ns;  // limit of every bounded wait in the kernel
  float out_scale;      // the last step's result is multiplied by it before the write
  int hold_signals;     // self-test only: never publish completions, so dependent items time out
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
  float *tile_partials;  // bf16 path: one sum of squares per 64x64 tile of W
  int *tile_ext;         // bf16 path: per 64x64 tile of Y, 1 + its last non-zero row and column (0: none)
  float *rscale;         // bf16 path: per matrix 1 / (||Y||_F + eps)
  float out_scale;       // to_user: the normalised matrix is multiplied by it
  int *status;           // device status word (debug bounds checks)
};

struct ResParams {
  const ResDesc *mats;
  int nmats;
  int cluster;           // CTAs per matrix (the launch's cluster size)
  int dtype;
  int steps;
  int ncoef;                        // 1: coef[0] for every step; else coef[step]
  float coef[kMaxTableSteps][3];    // (a, b, c)
  float eps;
  float out_scale;                  // the result is multiplied by it before the write
  int *status;                      // device status word (debug bounds checks)
};

// Momentum step of ns_muon_update_batched: up to kMomChunk matrices per launch.
constexpr int kMomChunk = 64;
struct MomentumParams {
  const void *g[kMomChunk];
  void *mom[kMomChunk];
  void *out[kMomChunk];
  int64_t numel[kMomChunk];
  int count;
  float mu;
  int nesterov;
  int *status;  // device status word (debug bounds checks)
};

constexpr int kNormBlocks = 128;  // partial-sum blocks per matrix
constexpr int kPrepTile = 64;     // Y tile edge of the preparation kernel

// tcgen05 GEMM tile (bf16 path). Tiles are processed by 2-CTA clusters: a
// tile list entry covers kTcPairM x kTcBN outputs, CTA rank r of the cluster
// computes rows [row0 + r*kTcBM, row0 + (r+1)*kTcBM) and loads half of the
// kTcBN-row second operand; the pair MMA reads both halves, so no operand
// byte is loaded twice.
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
int launch_split_prep(const PrepParams &p, int total_tiles, cudaStream_t s);
int launch_norm_tiles(const PrepParams &p, int total_tiles, int max_blocks, cudaStream_t s);
int launch_norm_finish(const PrepParams &p, cudaStream_t s);
int launch_resident(const ResParams &p, int smem_bytes, cudaStream_t s);
int launch_simt_phase(int phase, const PhaseParams &p, cudaStream_t s);
int launch_tc(const TcParams &p, int max_ctas, cudaStream_t s);
int tc_smem_bytes();
int launch_wait_probe(int *status, uint64_t limit_ns, int *gave_up, cudaStream_t s);
int launch_momentum(const MomentumParams &p, int dtype, int sms, cudaStream_t s);
int launch_bounds_probe(int *status, const void *base, cudaStream_t s);
int resident_smem_bytes(int m, int ns, int dtype, int cluster);  // one CTA of a matrix split over `cluster` CTAs
int resident_cluster(int m, int n);                 // CTAs per matrix of the resident kernel
int resident_slice(int n, int cluster);             // their slice width

void count_launch();

// The dynamic shared memory a kernel has been allowed on each device so far,
// so that the opt-in (cudaFuncSetAttribute) runs once per device and size
// rather than before every launch.
struct SmemOptIn {
  int allowed[64] = {};
  int ensure(const void *kernel, int bytes);  // 0, or -1 if the attribute could not be set
};

// Validation of a device-pointer call (the same checks, in the same order, as
// ns_orthogonalize_batched makes before launching) and the current-device
// check: NS_OK, or the status code such a call would return.
int check_call(void *const *X, const int64_t *shapes, int count, int steps, int dtype);

}  // namespace ns
