// ns_tc.cu -- bf16 tensor-core GEMM phases of libns on sm_103a (tcgen05).
//
// One persistent, warp-specialised kernel, launched as clusters of two CTAs
// over a sequence of work items: for every step, the gram tiles of all
// matrices, then the square tiles, then the apply tiles (each list largest
// ns_cost first); an item is one 256 x 256 output tile. By default the host
// launches the kernel once per step and phase, over that phase's items. In
// the single-launch schedule one launch runs every step and phase of the
// call: before loading an item's operands the producer waits until every item
// of the same matrix in earlier phases is complete (a per-matrix counter that
// the signal warp advances after the epilogue's stores), so the phases of
// different matrices overlap. Each tile is one pair MMA
// (tcgen05.mma.cta_group::2, M = 256, N = 256, K = 16, bf16 in, fp32
// accumulate) issued by the pair's leader CTA (rank 0): CTA rank r holds
// rows r*128 .. r*128+127 of the first operand and rows r*128 .. r*128+127 of
// the second in its own shared memory, and receives rows r*128 .. of the
// 256 x 256 accumulator in its own TMEM. No operand byte is loaded twice.
//   warp 0      TMA producer (both CTAs): its 128 x 64 share of each operand
//               per k-block (one 64 x 128 box K-major, or two 64 x 64 boxes
//               MN-major) into a 6-stage ring of 32 KB (128-byte swizzle);
//               the bytes of both CTAs are counted on the leader's full
//               barrier; the whole warp runs the loop, one elected lane issues;
//   warp 1      TMEM allocation (512 columns = two accumulators, cta_group::2)
//               in both CTAs; in the leader the warp runs the MMA loop and one
//               elected lane issues the pair MMAs and the commits that release
//               stages and hand accumulators to both CTAs' epilogues;
//   warps 2..9  epilogue (both CTAs): tcgen05.ld of its 128 accumulator rows
//               (two warps per TMEM lane quarter), the fused element-wise step
//               in fp32, round-to-nearest-even to bf16 and the stores; the
//               operand the step re-reads (A, or the iterate) is copied ahead
//               (cp.async) and the results leave through two swizzled 32 x 32
//               staging tiles per warp, so that every global access of the
//               warp moves 8 rows x 64 contiguous bytes; the second
//               accumulator lets the next tile's main loop overlap it;
//   warp 10     publishes each stored item on its matrix's completion counter.
// Phases (see ns_internal.h for the layout). Iterates stay in the caller's
// orientation; step 0 reads the caller's Y directly when TMA can address it.
//   0 gram    A = W W^T             upper-triangle tiles, each stored whole (no
//                                   mirror); operands MN-major when transposed
//   1 square  B = b A + c (A A)     upper-triangle tiles, each stored whole; A's
//                                   rows left of the diagonal read MN-major from
//                                   the mirrored upper tiles
//   2 apply   W' = a W + B W        tiles of the next iterate in the caller's
//                                   orientation (B W, or W^T B when transposed;
//                                   B's rows left of the diagonal read MN-major),
//                                   one straight store (the caller's Y on the last step)
// Tiles wholly outside a matrix's non-zero extent are skipped, and k-loops
// stop at the extent: zero rows and columns stay zero through every step.
// Every wait is bounded (see mbar_wait); a timeout sets the status word and
// the CTA drains its in-flight copies and MMAs, frees TMEM and exits.
#include <cuda_runtime.h>

#include "ns_device.cuh"

namespace ns {

namespace {

constexpr int kEpiWarps = 8;                        // two per TMEM lane quarter
constexpr int kSignalWarp = 2 + kEpiWarps;          // publishes item completion GPU-wide
constexpr int kThreads = 32 * (kSignalWarp + 1);    // producer, MMA, epilogue warps, signal warp
constexpr int kChunksPerWarp = (kTcBN / 32) / (kEpiWarps / 4);
// per-warp staging tiles of the epilogue's coalesced loads and stores: 32 rows
// of 32 bf16 (16 words), the four 16-byte pieces of a row permuted by an XOR
// swizzle (see stage_word)
constexpr int kRowStageWords = 16;
constexpr int kStageTileWords = 32 * kRowStageWords;
constexpr int kEpiStageBytes = 2 * kStageTileWords * 4;  // two tiles per warp
constexpr int kStages = 6;
constexpr int kABytes = kTcBM * kTcBK * 2;          // 16 KB: this CTA's 128 rows of the first operand
constexpr int kBBytes = (kTcBN / 2) * kTcBK * 2;    // 16 KB: this CTA's half of the second operand
constexpr int kStageBytes = kABytes + kBBytes;      // 32 KB per CTA
constexpr int kPairStageBytes = 2 * kStageBytes;    // both CTAs' loads, counted at the leader
constexpr int kBoxBytes = 64 * 64 * 2;             // one TMA box: 64 x 64 bf16
static_assert(kABytes == 2 * kBoxBytes && kBBytes == 2 * kBoxBytes, "operand share = two boxes");
constexpr int kAccs = 2;                            // accumulators (each kTcBN TMEM columns)
constexpr int kTmemCols = kAccs * kTcBN;

// One work item as the pair's fetcher decodes it: item index (p.g_end: no
// more items), step, phase and the matrix's orientation (packed), tile
// record and the matrix's extents. The fetcher (the leader CTA's producer
// warp) publishes each item of the pair, in order, into a small queue in both
// CTAs' shared memory; every other role of both CTAs takes its items from
// that queue, so all roles see the same sequence and none of them waits on a
// global lookup.
struct QItem {
  int g;
  int spf;               // step * 16 + phase * 4 + transposed * 2 + direct
  int mat, row0, col0;
  int e0, e1;
  int pad;
  __device__ int step() const { return spf >> 4; }
  __device__ int phase() const { return (spf >> 2) & 3; }
  __device__ int tr() const { return (spf >> 1) & 1; }
  __device__ int direct() const { return spf & 1; }
};
static_assert(sizeof(QItem) == 32, "two 16-byte words");
constexpr int kQueue = 8;  // published items a pair may run ahead of its slowest role
// consumers that release a queue slot: in the leader the MMA warp, the
// epilogue warps and the signal warp; in the peer its producer warp, epilogue
// warps and signal warp
constexpr int kQueueConsumers = 2 * (kEpiWarps + 2);

struct Barriers {
  QItem queue[kQueue];      // each CTA: the pair's items in order (written by the leader's fetcher)
  uint64_t qfull[kQueue];   // each CTA: a queue slot holds the next item
  uint64_t qempty[kQueue];  // leader: every consumer of both CTAs has read a slot
  uint64_t full[kStages];   // leader: both CTAs' loads of a stage landed
  uint64_t empty[kStages];  // each CTA: the leader's MMAs are done with a stage
  uint64_t tfull[2];        // each CTA: an accumulator is ready
  uint64_t tempty[2];       // leader: every epilogue warp of both CTAs is done with an accumulator
  uint64_t epi_done[2];     // each CTA: its epilogue warps stored an item (signal warp waits on it)
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

constexpr int kBarrierBytes = (static_cast<int>(sizeof(Barriers)) + 127) / 128 * 128;

struct TileInfo {
  const MatDesc *d;
  int mat;
  int row0, col0;
  int nk;
  int tr;  // the matrix is transposed (M > N)
  bool skip;
};

// Item g of the launch's sequence: step, phase and tile index in that phase's list.
__device__ __forceinline__ void decode_item(const TcParams &p, int g, int &step, int &phase, int &t) {
  const int per_step = 2 * p.n01 + p.n2;
  step = g / per_step;
  const int r = g - step * per_step;
  phase = r < p.n01 ? 0 : (r < 2 * p.n01 ? 1 : 2);
  t = phase == 0 ? r : (phase == 1 ? r - p.n01 : r - 2 * p.n01);
}

// Tile info from the tile record, the matrix's extents and its orientation.
__device__ __forceinline__ TileInfo make_tile_info(const TcParams &p, int phase, const Tile &tl, int e0, int e1,
                                                   int tr) {
  TileInfo ti;
  ti.mat = tl.mat;
  ti.d = p.mats + tl.mat;
  ti.row0 = tl.row0;
  ti.col0 = tl.col0;
  ti.tr = tr;
  const int meff = tr ? e1 : e0, neff = tr ? e0 : e1;
  const int k_eff = phase == 0 ? neff : meff;
  // decided per pair tile, so both CTAs of a cluster agree; gram and square
  // tiles are over m x m, apply tiles over the caller's M x N
  ti.skip = phase == 2 ? (tl.row0 >= e0) || (tl.col0 >= e1) : (tl.row0 >= meff) || (tl.col0 >= meff);
  ti.nk = (k_eff + kTcBK - 1) / kTcBK;
  return ti;
}


// The item sequence of one pair as its fetcher produces it: indices from the
// call's ticket counter (single-launch schedule: every pair takes the lowest
// item not yet taken, so the items in flight stay contiguous), or the pair's
// static stride (one launch per phase). The lookups run ahead of use: while
// an item is produced, the matrix record of the next item, the tile record of
// the one after and the ticket of the one after that are in flight.
struct Fetcher {
  int g, sp;               // the item to publish next: index, step * 16 + phase * 4
  Tile tl;                 // its tile record
  int e0, e1, tr, direct;  // its matrix's extents and orientation
  int g2, sp2;             // the item after it
  Tile tl2;                // and its tile record
  int pending;             // lane 0: the raw ticket of the item after g2 (ticket mode)
};
// Only loaded values are carried in the fetcher; arithmetic on them waits
// until the item is published, so no lookup stalls the warp before its use.

__device__ __forceinline__ Tile fetch_tile(const TcParams &p, int g, int &sp) {
  int step, phase, t;
  decode_item(p, g, step, phase, t);
  sp = step * 16 + phase * 4;
  return (phase < 2 ? p.tiles01 : p.tiles2)[t];
}

__device__ __forceinline__ void fetch_matrix(const TcParams &p, Fetcher &f) {
  const MatDesc &d = p.mats[f.tl.mat];
  f.e0 = p.ext[2 * f.tl.mat];
  f.e1 = p.ext[2 * f.tl.mat + 1];
  f.tr = d.transposed;
  f.direct = d.direct;
}

__device__ __forceinline__ int take_ticket(const TcParams &p) {
  return (threadIdx.x & 31) == 0 ? atomicAdd(p.ticket, 1) : 0;
}
__device__ __forceinline__ int clamp_item(const TcParams &p, int g) { return g < p.g_end ? g : p.g_end; }

// Whole warp: the first two items of the pair and the ticket of the third.
__device__ __forceinline__ void fetcher_start(const TcParams &p, int first, int stride, Fetcher &f) {
  if (p.tickets) {
    f.g = clamp_item(p, p.g_begin + __shfl_sync(0xffffffffu, take_ticket(p), 0));
    f.g2 = clamp_item(p, p.g_begin + __shfl_sync(0xffffffffu, take_ticket(p), 0));
    f.pending = take_ticket(p);
  } else {
    f.g = clamp_item(p, first);
    f.g2 = f.g < p.g_end ? clamp_item(p, f.g + stride) : p.g_end;
    f.pending = 0;
  }
  if (f.g < p.g_end) {
    f.tl = fetch_tile(p, f.g, f.sp);
    fetch_matrix(p, f);
  }
  if (f.g2 < p.g_end) f.tl2 = fetch_tile(p, f.g2, f.sp2);
}

// The item to publish, packed.
__device__ __forceinline__ QItem fetcher_item(const Fetcher &f) {
  QItem it;
  it.g = f.g;
  it.spf = f.sp | (f.tr << 1) | f.direct;
  it.mat = f.tl.mat;
  it.row0 = f.tl.row0;
  it.col0 = f.tl.col0;
  it.e0 = f.e0;
  it.e1 = f.e1;
  it.pad = 0;
  return it;
}

// Whole warp, right after the current item was published: the next item
// becomes current (its matrix record requested now, needed when it is
// published), the one after gets its index and tile record requested.
__device__ __forceinline__ void fetcher_advance(const TcParams &p, int stride, Fetcher &f) {
  f.g = f.g2;
  if (f.g >= p.g_end) return;
  f.sp = f.sp2;
  f.tl = f.tl2;
  fetch_matrix(p, f);
  if (p.tickets) {
    f.g2 = clamp_item(p, p.g_begin + __shfl_sync(0xffffffffu, f.pending, 0));
    f.pending = take_ticket(p);
  } else {
    f.g2 = clamp_item(p, f.g + stride);
  }
  if (f.g2 < p.g_end) f.tl2 = fetch_tile(p, f.g2, f.sp2);
}

// ---- the pair's item queue
__device__ __forceinline__ void st_cluster_v4(uint32_t addr, const uint4 &v) {
  asm volatile("st.shared::cluster.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

// The fetcher's lane publishes item number k of the pair into slot k % kQueue
// of both CTAs, once every consumer has read what the slot held before.
__device__ __forceinline__ bool queue_put(Barriers *bar, int k, const QItem &it, const Waiter &w) {
  const int slot = k % kQueue;
  const uint32_t parity = static_cast<uint32_t>(k / kQueue) & 1u;
  if (!mbar_wait<true>(&bar->qempty[slot], parity ^ 1u, w)) return false;
  const uint4 *v = reinterpret_cast<const uint4 *>(&it);
  uint4 *mine = reinterpret_cast<uint4 *>(&bar->queue[slot]);
  const uint32_t peer = mapa_shared(smem_u32(&bar->queue[slot]), 1);
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    mine[q] = v[q];
    st_cluster_v4(peer + 16 * q, v[q]);
  }
  mbar_arrive(&bar->qfull[slot]);                                   // release: this CTA's copy
  mbar_arrive_cluster(mapa_shared(smem_u32(&bar->qfull[slot]), 1));  // release.cluster: the peer's copy
  return true;
}

// Release slot k % kQueue on the leader: a relaxed arrive (a consumer only
// read the slot, and calls this after it has used what it read, so no fence
// has to wait for its own earlier stores).
__device__ __forceinline__ void queue_release(Barriers *bar, int k) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(
                   mapa_shared(smem_u32(&bar->qempty[k % kQueue]), 0))
               : "memory");
}

// One lane takes item number k of the pair from its CTA's queue (the caller
// releases the slot once it has used the item).
__device__ __forceinline__ bool queue_get_lane(Barriers *bar, int k, QItem &it, const Waiter &w) {
  const int slot = k % kQueue;
  const uint32_t parity = static_cast<uint32_t>(k / kQueue) & 1u;
  if (!mbar_wait<true>(&bar->qfull[slot], parity, w)) return false;
  const volatile uint4 *src = reinterpret_cast<const volatile uint4 *>(&bar->queue[slot]);
  uint4 *dst = reinterpret_cast<uint4 *>(&it);
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const uint4 v = make_uint4(src[q].x, src[q].y, src[q].z, src[q].w);
    dst[q] = v;
  }
  return true;
}

// The same for a whole warp: lane 0 takes the item, broadcasts it (which
// uses what it read) and releases the slot.
__device__ __forceinline__ bool queue_get_warp(Barriers *bar, int k, QItem &it, const Waiter &w) {
  int ok = 1;
  if ((threadIdx.x & 31) == 0) ok = queue_get_lane(bar, k, it, w) ? 1 : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  int *v = reinterpret_cast<int *>(&it);
#pragma unroll
  for (int q = 0; q < 7; ++q) v[q] = __shfl_sync(0xffffffffu, v[q], 0);
  if (ok && (threadIdx.x & 31) == 0) queue_release(bar, k);
  return ok != 0;
}

__device__ __forceinline__ TileInfo item_info(const TcParams &p, const QItem &it) {
  return make_tile_info(p, it.phase(), Tile{it.mat, it.row0, it.col0, 0}, it.e0, it.e1, it.tr());
}

__device__ __forceinline__ TileInfo tile_info(const TcParams &p, int phase, int t) {
  const Tile tl = (phase < 2 ? p.tiles01 : p.tiles2)[t];
  return make_tile_info(p, phase, tl, p.ext[2 * tl.mat], p.ext[2 * tl.mat + 1], p.mats[tl.mat].transposed);
}

// Per-phase launches: the items of one pair (g, g + stride, ...), which
// every role computes for itself, with their global lookups pipelined, for
// the single-thread roles whose every stall idles the tensor pipe: while an item runs, the tile record of the item after next and the
// extents and orientation of the next item are already being loaded. Only
// loaded values are carried; arithmetic on them waits until the item is taken.
struct ItemPipe {
  int g;                   // item taken next
  int step, phase;         // of item g
  Tile tl;                 // of item g
  int e0, e1, tr, direct;  // of item g's matrix
  int step2, phase2;       // of item g + stride
  Tile tl2;                // of item g + stride
};

__device__ __forceinline__ Tile fetch_tile_sp(const TcParams &p, int g, int &step, int &phase) {
  int t;
  decode_item(p, g, step, phase, t);
  return (phase < 2 ? p.tiles01 : p.tiles2)[t];
}

__device__ __forceinline__ void fetch_matrix_sp(const TcParams &p, ItemPipe &q) {
  const MatDesc &d = p.mats[q.tl.mat];
  q.e0 = p.ext[2 * q.tl.mat];
  q.e1 = p.ext[2 * q.tl.mat + 1];
  q.tr = d.transposed;
  q.direct = d.direct;
}

__device__ __forceinline__ void pipe_start(const TcParams &p, int g, int stride, ItemPipe &q) {
  q.g = g;
  if (g < p.g_end) {
    q.tl = fetch_tile_sp(p, g, q.step, q.phase);
    fetch_matrix_sp(p, q);
  }
  if (g + stride < p.g_end) q.tl2 = fetch_tile_sp(p, g + stride, q.step2, q.phase2);
}

// Take item q.g (returned through step, phase, ti) and start the lookups of the two after it.
__device__ __forceinline__ void pipe_take(const TcParams &p, int stride, ItemPipe &q, int &step, int &phase,
                                          TileInfo &ti, int &direct) {
  step = q.step;
  phase = q.phase;
  ti = make_tile_info(p, q.phase, q.tl, q.e0, q.e1, q.tr);
  direct = q.direct;
  q.g += stride;
  if (q.g < p.g_end) {
    q.step = q.step2;
    q.phase = q.phase2;
    q.tl = q.tl2;
    fetch_matrix_sp(p, q);
  }
  if (q.g + stride < p.g_end) q.tl2 = fetch_tile_sp(p, q.g + stride, q.step2, q.phase2);
}

// The k-loop of an item as three consecutive k-ranges with a fixed operand
// order each: [0, e0) both operands MN-major, [e0, e1) the first K-major and
// the second MN-major, [e1, nk) both K-major (any of them may be empty).
// map[o][0] / map[o][1] are the tensor maps of the first (A, rows of the
// tile) and second (B, columns of the tile) operand in range o.
//
// The symmetric products A and B are stored as their upper 256 x 256 tiles
// only (every element of each, diagonal tiles included): an operand's rows
// in tile row X are read K-major from the stored tiles (X, K) for k-blocks of
// tile column K >= X, and MN-major from the mirrored stored tiles (K, X) for
// K < X (A = A^T).
struct ItemPlan {
  int e0, e1;
  const void *map[3][2];
};

__device__ __forceinline__ ItemPlan plan_item(const MatDesc &d, int step, int phase, int transposed, int direct,
                                              int row0, int col0, int nk) {
  // the iterate read at this step: Y itself or its copy on step 0, then the
  // ping-pong buffers; each has a K-major and an MN-major map
  const bool y = step == 0 && direct;
  const void *src_k = y ? &d.tm_y : &d.tm_s[step & 1];
  const void *src_mn = y ? &d.tm_y_mn : &d.tm_s_mn[step & 1];
  const int kb_row = min(row0 / kTcBK, nk), kb_col = min(col0 / kTcBK, nk);  // the diagonal tile's first k-block
  ItemPlan pl;
  if (phase == 0) {  // W W^T from the iterate: W's rows are its columns when transposed
    pl.e0 = pl.e1 = transposed ? nk : 0;
    pl.map[0][0] = pl.map[0][1] = src_mn;
    pl.map[1][0] = pl.map[1][1] = src_mn;
    pl.map[2][0] = pl.map[2][1] = src_k;
  } else if (phase == 1) {  // A A: both operands from A's upper tiles (row0 <= col0)
    pl.e0 = kb_row;
    pl.e1 = max(kb_row, kb_col);
    pl.map[0][0] = pl.map[0][1] = &d.tm_a_mn;
    pl.map[1][0] = &d.tm_a;
    pl.map[1][1] = &d.tm_a_mn;
    pl.map[2][0] = pl.map[2][1] = &d.tm_a;
  } else if (transposed) {  // W^T B: iterate rows (K-major) times B's rows col0..
    pl.e0 = 0;
    pl.e1 = kb_col;
    pl.map[0][0] = src_mn;  // (unused: empty range)
    pl.map[0][1] = &d.tm_b_mn;
    pl.map[1][0] = src_k;
    pl.map[1][1] = &d.tm_b_mn;
    pl.map[2][0] = src_k;
    pl.map[2][1] = &d.tm_b;
  } else {  // B W: B's rows row0.. times the iterate's columns (MN-major)
    pl.e0 = kb_row;
    pl.e1 = nk;
    pl.map[0][0] = &d.tm_b_mn;
    pl.map[0][1] = src_mn;
    pl.map[1][0] = &d.tm_b;
    pl.map[1][1] = src_mn;
    pl.map[2][0] = &d.tm_b;  // (unused: empty range)
    pl.map[2][1] = src_mn;
  }
  return pl;
}

// Prefetch the tensor maps an item of (step, phase) of matrix d may read, so
// a tile start does not wait for its descriptors (consecutive items of a
// pair often belong to different matrices). Only the maps' addresses are
// formed: nothing of d is read, so this does not wait for its record.
__device__ __forceinline__ void prefetch_item_maps(const MatDesc &d, int step, int phase) {
  if (phase == 1) {
    prefetch_tensormap(&d.tm_a);
    prefetch_tensormap(&d.tm_a_mn);
    return;
  }
  if (phase == 2) {
    prefetch_tensormap(&d.tm_b);
    prefetch_tensormap(&d.tm_b_mn);
  }
  prefetch_tensormap(&d.tm_s[step & 1]);
  prefetch_tensormap(&d.tm_s_mn[step & 1]);
  if (step == 0) {
    prefetch_tensormap(&d.tm_y);
    prefetch_tensormap(&d.tm_y_mn);
  }
}

// The same for an item whose matrix record is known: exactly the maps it reads.
__device__ __forceinline__ void prefetch_item_maps_exact(const MatDesc &d, int step, int phase, int transposed,
                                                         int direct) {
  const bool y = step == 0 && direct;
  const void *src_k = y ? &d.tm_y : &d.tm_s[step & 1];
  const void *src_mn = y ? &d.tm_y_mn : &d.tm_s_mn[step & 1];
  if (phase == 0) {
    prefetch_tensormap(transposed ? src_mn : src_k);
  } else if (phase == 1) {
    prefetch_tensormap(&d.tm_a);
    prefetch_tensormap(&d.tm_a_mn);
  } else {
    prefetch_tensormap(&d.tm_b);
    prefetch_tensormap(&d.tm_b_mn);
    prefetch_tensormap(transposed ? src_k : src_mn);
  }
}

// TMA of one operand share: 128 tile rows [mn0, mn0 + 128) by K [k0, k0 + 64).
// K-major: one box of 128 rows. MN-major: box rows are K indices and the tile
// index runs along them, 64 per box row, so two 64 x 64 boxes 8 KB apart.
// MN is a template parameter so the producer issues only the copies it needs.
// kSplit: the tensor is three bf16 slices behind a 3-D map, z the slice.
template <int MN, int kSplit>
__device__ __forceinline__ void load_operand(uint8_t *dst, const void *map, int mn0, int k0, int z,
                                             uint32_t bar_cluster, uint64_t pol) {
  if (kSplit) {
    if (MN) {
      tma_load_3d_pair(dst, map, mn0, k0, z, bar_cluster, pol);
      tma_load_3d_pair(dst + kBoxBytes, map, mn0 + 64, k0, z, bar_cluster, pol);
    } else {
      tma_load_3d_pair(dst, map, k0, mn0, z, bar_cluster, pol);
    }
  } else if (MN) {
    tma_load_2d_pair(dst, map, mn0, k0, bar_cluster, pol);
    tma_load_2d_pair(dst + kBoxBytes, map, mn0 + 64, k0, bar_cluster, pol);
  } else {
    tma_load_2d_pair(dst, map, k0, mn0, bar_cluster, pol);
  }
}

// fp32 path: every tensor W, A, B is held as three bf16 slices x = h + m + l
// (h = bf16(x), m = bf16(x - h), l = bf16(x - h - m): 24 significant bits),
// and a product X Y is the sum of the six slice products whose weights are
// at least 2^-18 of the leading one -- (h,h), (h,m), (m,h), (h,l), (l,h),
// (m,m) -- accumulated in one fp32 accumulator; the dropped three weigh
// 2^-27 or less. Part p of an item multiplies slice part_a(p) of the first
// operand by slice part_b(p) of the second over the whole k range. The parts
// run smallest first: the tensor core's accumulation loses up to about one
// unit in the last place of the running sum per instruction, so the small
// parts, added while the sum is still ~2^-9 of its final size, contribute
// almost nothing to the error, and only the (h,h) pass adds at full size.
constexpr int kSplitParts = 6;
__host__ __device__ constexpr int part_a(int part) { return (0x010120 >> (4 * part)) & 15; }  // 0 2 1 0 1 0
__host__ __device__ constexpr int part_b(int part) { return (0x001102 >> (4 * part)) & 15; }  // 2 0 1 1 0 0
static_assert(part_a(0) == 0 && part_b(0) == 2 && part_a(1) == 2 && part_b(1) == 0 && part_a(2) == 1 &&
                  part_b(2) == 1 && part_a(3) == 0 && part_b(3) == 1 && part_a(4) == 1 && part_b(4) == 0 &&
                  part_a(5) == 0 && part_b(5) == 0,
              "slice pairs (h,l) (l,h) (m,m) (h,m) (m,h) (h,h)");

// Operand descriptor of the share at `addr` for K sub-step kk (16 K each).
template <int MN>
__device__ __forceinline__ uint64_t operand_desc(uint32_t addr, int kk) {
  return MN ? sw128_mnmajor_desc(addr + static_cast<uint32_t>(kk) * 2048u)
            : sw128_kmajor_desc(addr + static_cast<uint32_t>(kk) * 32u);
}

// The iterate read at `step` (the caller's Y or a workspace buffer) and its pitch.
__device__ __forceinline__ const __nv_bfloat16 *iterate_src(const MatDesc &d, int step, int &pitch) {
  if (step == 0 && d.direct) {
    pitch = d.N;
    return static_cast<const __nv_bfloat16 *>(d.user);
  }
  pitch = d.ps;
  return static_cast<const __nv_bfloat16 *>(d.s[step & 1]);
}

// The signal warp of each CTA advances a matrix's counter by one per item,
// computed or skipped, and only after the item's own dependencies are met
// (a computed item after its epilogue stored it); hence
// counter >= units_before(step, phase) implies that every earlier item of the
// matrix is complete.
constexpr int kUnitsPerItem = kTcCluster;

// Counter value at which every item of matrix d in phases before (step, phase) is complete.
__device__ __forceinline__ int units_before(const MatDesc &d, int step, int phase) {
  const int items = step * (2 * d.t01 + d.t2) + (phase >= 1 ? d.t01 : 0) + (phase >= 2 ? d.t01 : 0);
  return kUnitsPerItem * items;
}

// Per-item constants of the epilogue.
struct StepCtx {
  int *status;      // device status word (debug bounds checks)
  int step;
  int final_step;   // apply writes the caller's matrix
  float ca, cb, cc;
  float gs, as;     // step 0 folds the normalisation in: A *= r^2, W' *= r (else 1);
                    // the last step also applies the output scale
};

__device__ __forceinline__ StepCtx step_ctx(const TcParams &p, int step, int mat) {
  const float *co = p.coef[p.ncoef == 1 ? 0 : step];
  StepCtx c;
  c.status = p.status;
  c.step = step;
  c.final_step = step == p.steps - 1;
  c.ca = co[0];
  c.cb = co[1];
  c.cc = co[2];
  const float r = (step == 0 && p.rscale) ? p.rscale[mat] : 1.0f;
  c.gs = r * r;
  c.as = c.final_step ? r * p.out_scale : r;
  return c;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t *>(&v);
}

// Writes 8 bf16 (one 16-byte word, `o`) at dst = row R, columns C0..C0+7,
// keeping only elements with column < col_lim and, when upper, column >= R.
// The destination buffer of a store: where it starts and how many bytes it
// has (debug builds check every store against it).
struct StoreBuf {
  const void *base;
  size_t bytes;
  int *status;
};

__device__ __forceinline__ void store_piece8(__nv_bfloat16 *dst, const uint4 &o, int R, int C0, int col_lim,
                                             bool upper, const StoreBuf &sb) {
  const bool all = (C0 + 8 <= col_lim) && (!upper || C0 >= R) && ((reinterpret_cast<uintptr_t>(dst) & 15) == 0);
  if (all) {
    if (in_bounds(dst, 16, sb.base, sb.bytes, sb.status)) *reinterpret_cast<uint4 *>(dst) = o;
    return;
  }
  const uint32_t w[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const int C = C0 + e;
    if (C < col_lim && (!upper || C >= R) && in_bounds(dst + e, 2, sb.base, sb.bytes, sb.status))
      dst[e] = __ushort_as_bfloat16(static_cast<uint16_t>(w[e >> 1] >> (16 * (e & 1))));
  }
}

// Word offset of 16-byte piece `piece` (0..3) of row `row` (0..31) in a warp's
// staging tile. The block moves between two layouts: one row per lane (lane l
// holds row l), and coalesced (in access k, lane l holds piece l % 4 of row
// 8k + l / 4, so that 8 rows x 64 contiguous bytes of global memory move per
// instruction). A 16-byte shared-memory access is served eight lanes at a
// time; XOR-ing the piece index with bits 1..2 of the row puts the eight
// lanes of either layout on 32 different banks.
__device__ __forceinline__ int stage_word(int row, int piece) {
  return row * kRowStageWords + 4 * (piece ^ ((row >> 1) & 3));
}

// Warp-cooperative store of a 32 x 32 block held one row per lane: lane l
// holds v[t] = element (row row0 + l, column col0 + t). The rows go through
// the warp's staging tile so that each store instruction writes 8 rows x 64
// contiguous bytes (4 lanes per row). Elements are written only where
// row < row_lim, column < col_lim and, if upper, column >= row.
__device__ __forceinline__ void warp_store_rows(uint32_t *stage, const float (&v)[32], __nv_bfloat16 *base,
                                                size_t pitch, int row0, int row_lim, int col0, int col_lim,
                                                bool upper, int *status) {
  // the buffer: row_lim rows of `pitch` elements
  const StoreBuf sb{base, static_cast<size_t>(row_lim) * pitch * 2, status};
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int q = 0; q < 4; ++q)
    *reinterpret_cast<uint4 *>(stage + stage_word(lane, q)) =
        make_uint4(pack_bf16x2(v[8 * q + 0], v[8 * q + 1]), pack_bf16x2(v[8 * q + 2], v[8 * q + 3]),
                   pack_bf16x2(v[8 * q + 4], v[8 * q + 5]), pack_bf16x2(v[8 * q + 6], v[8 * q + 7]));
  __syncwarp();
  const int piece = lane & 3;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int rl = 8 * k + (lane >> 2);
    const int R = row0 + rl;
    if (R < row_lim) {
      const uint4 o = *reinterpret_cast<const uint4 *>(stage + stage_word(rl, piece));
      store_piece8(base + static_cast<size_t>(R) * pitch + col0 + 8 * piece, o, R, col0 + 8 * piece, col_lim, upper,
                   sb);
    }
  }
  __syncwarp();
}

// The global operand an epilogue reads besides the accumulator (A for square,
// the current iterate for apply) over the warp's 32 rows of an item: where
// its row r0 .. r0+31, column ti.col0 starts and its row pitch, or nullptr
// when those rows are not all inside the matrix; chunks (32-column blocks)
// below col_lim lie wholly inside it. Elements of the other blocks are read
// one by one by epilogue_chunk.
struct OperandRows {
  const __nv_bfloat16 *base;
  int pitch;
  int col_lim;
  __device__ __forceinline__ const __nv_bfloat16 *block(int chunk) const {
    return (base && chunk * 32 + 32 <= col_lim) ? base + chunk * 32 : nullptr;
  }
};

template <int PHASE>
__device__ __forceinline__ OperandRows operand_rows(const StepCtx &p, const TileInfo &ti, int r) {
  const MatDesc &d = *ti.d;
  const int row = ti.row0 + (r & ~31);
  OperandRows o;
  if (PHASE == 1) {
    o.pitch = d.pm;
    o.col_lim = d.m - ti.col0;
    o.base = row + 32 <= d.m
                 ? static_cast<const __nv_bfloat16 *>(d.a) + static_cast<size_t>(row) * d.pm + ti.col0
                 : nullptr;
  } else {
    const __nv_bfloat16 *S = iterate_src(d, p.step, o.pitch);
    o.col_lim = d.N - ti.col0;
    o.base = row + 32 <= d.M ? S + static_cast<size_t>(row) * o.pitch + ti.col0 : nullptr;
  }
  return o;
}

// Fetches a chunk's operand block ahead of time into a staging tile of the
// warp, coalesced and without registers: in access k lane l copies piece
// l % 4 (8 bf16) of block row 8k + l / 4 (cp.async, through L2 only), so each
// access of the warp reads 8 rows x 64 contiguous bytes. Nothing is copied
// when the block is not whole. One commit group per call and lane.
__device__ __forceinline__ void fetch_chunk(const OperandRows &op, int chunk, uint32_t *tile) {
  const __nv_bfloat16 *blk = op.block(chunk);
  const int lane = threadIdx.x & 31;
  if (blk) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int row = 8 * k + (lane >> 2), piece = lane & 3;
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(tile + stage_word(row, piece))),
                   "l"(blk + static_cast<size_t>(row) * op.pitch + 8 * piece)
                   : "memory");
    }
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
}

// Waits until at most N of this lane's fetch_chunk groups are in flight.
template <int N>
__device__ __forceinline__ void fetch_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// A block fetched by fetch_chunk reaches one row per lane through the
// staging tile: staged_row gives lane l the 32 elements (packed, 8 per word)
// of block row l.
__device__ __forceinline__ void staged_row(const uint32_t *stage, uint4 (&w4)[4]) {
  const int lane = threadIdx.x & 31;
  __syncwarp();
#pragma unroll
  for (int q = 0; q < 4; ++q) w4[q] = *reinterpret_cast<const uint4 *>(stage + stage_word(lane, q));
  __syncwarp();
}

// The first n (0..32) bf16 of src, zero beyond, packed as staged_row packs a row.
__device__ __forceinline__ void gather_row(const __nv_bfloat16 *src, int n, uint4 (&w4)[4]) {
  uint32_t w[16];
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    const uint32_t lo = 2 * e < n ? __bfloat16_as_ushort(src[2 * e]) : 0u;
    const uint32_t hi = 2 * e + 1 < n ? __bfloat16_as_ushort(src[2 * e + 1]) : 0u;
    w[e] = lo | (hi << 16);
  }
#pragma unroll
  for (int q = 0; q < 4; ++q) w4[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
}

// Element t (0..31) of a packed row.
__device__ __forceinline__ float row_elem(const uint4 (&w4)[4], int t) {
  const uint4 &q = w4[t >> 3];
  const uint32_t w = ((t >> 1) & 3) == 0 ? q.x : ((t >> 1) & 3) == 1 ? q.y : ((t >> 1) & 3) == 2 ? q.z : q.w;
  return __uint_as_float((t & 1) ? (w & 0xffff0000u) : (w << 16));
}

// Epilogue of one 32-column chunk held by one thread: tile row r, columns
// chunk*32 .. chunk*32+31 of the tile. When the chunk's operand block is
// whole (`staged`) it is already in the staging tile `stage` (fetch_chunk).
template <int PHASE>
__device__ __forceinline__ void epilogue_chunk(const StepCtx &p, const TileInfo &ti, int r, int chunk,
                                               const uint32_t (&raw)[32], bool staged, uint32_t *stage) {
  const MatDesc &d = *ti.d;
  const int r0 = r & ~31;  // the warp's first tile row
  float f[32];
#pragma unroll
  for (int t = 0; t < 32; ++t) f[t] = __uint_as_float(raw[t]);

  if (PHASE == 0 || PHASE == 1) {
    const int m = d.m, pm = d.pm;
    const int i = ti.row0 + r;
    const int i0 = ti.row0 + r0;
    const int jb = ti.col0 + chunk * 32;
    // warp-uniform: the whole 32x32 block is outside the matrix
    if (i0 >= m || jb >= m) return;
    if (PHASE == 0) {
#pragma unroll
      for (int t = 0; t < 32; ++t) f[t] *= p.gs;  // A = r^2 Y Y^T on the first step
    }
    const bool mine = i < m;
    if (PHASE == 1) {
      const __nv_bfloat16 *A = static_cast<const __nv_bfloat16 *>(d.a) + static_cast<size_t>(i) * pm + jb;
      uint4 aold[4];
      if (staged)  // warp-uniform
        staged_row(stage, aold);
      else
        gather_row(A, mine ? min(32, m - jb) : 0, aold);
#pragma unroll
      for (int t = 0; t < 32; ++t) f[t] = p.cb * row_elem(aold, t) + p.cc * f[t];
    }
    // the whole upper tile (both halves of a diagonal tile); readers take the
    // lower triangle from the mirrored upper tiles
    __nv_bfloat16 *O = static_cast<__nv_bfloat16 *>(PHASE == 0 ? d.a : d.b);
    warp_store_rows(stage, f, O, pm, i0, m, jb, m, false, p.status);
  } else {
    // tile rows R over the caller's M, columns C over N
    const int M = d.M, N = d.N;
    const int R = ti.row0 + r;
    const int R0 = ti.row0 + r0;         // the warp's first row
    const int C = ti.col0 + chunk * 32;
    if (R0 >= M || C >= N) return;       // warp-uniform
    const bool mine = R < M;
    int sp;
    const __nv_bfloat16 *S = iterate_src(d, p.step, sp);
    S += static_cast<size_t>(R) * sp + C;
    uint4 xo[4];
    if (staged)  // warp-uniform
      staged_row(stage, xo);
    else
      gather_row(S, mine ? min(32, N - C) : 0, xo);
#pragma unroll
    for (int t = 0; t < 32; ++t) f[t] = p.as * (p.ca * row_elem(xo, t) + f[t]);  // r (a Y + B Y) on the first step
    if (!p.final_step)
      warp_store_rows(stage, f, static_cast<__nv_bfloat16 *>(d.s[(p.step + 1) & 1]), static_cast<size_t>(d.ps), R0,
                      M, C, N, false, p.status);
    else
      warp_store_rows(stage, f, static_cast<__nv_bfloat16 *>(d.user), static_cast<size_t>(N), R0, M, C, N, false,
                      p.status);
  }
}

// Bounded wait that ignores the abort flag: used only to drain in-flight
// asynchronous work before the CTA releases its shared memory and TMEM.
__device__ __forceinline__ void mbar_drain(uint64_t *bar, uint32_t parity, const Waiter &w) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > w.limit_ns) {
      set_status(w.status, kStatusTimeout);
      return;
    }
  }
}



// Epilogue of one item in one epilogue warp: prefetch the operand it
// reloads, wait for the accumulator, then drain this warp's chunks.
template <int PHASE>
__device__ __forceinline__ bool epilogue_item(const StepCtx &sc, const TileInfo &ti, int r, int c0, uint32_t tbase,
                                              uint32_t *stage, uint64_t *tfull, uint32_t parity, const Waiter &w) {
  // the operand does not depend on the accumulator: fetch it while the MMAs run
  // staging tiles: chunk c0 + k uses tile k % 2 for its operand block and its stores
  uint32_t *tiles[2] = {stage, stage + kStageTileWords};
  OperandRows op{};
  if (PHASE != 0) {
    op = operand_rows<PHASE>(sc, ti, r);
    fetch_chunk(op, c0, tiles[0]);
    fetch_chunk(op, c0 + 1, tiles[1]);
  }
  if (!mbar_wait<true>(tfull, parity, w)) {
    fetch_wait<0>();  // no copy into the staging tiles outlives the item
    return false;
  }
  tc_fence_after();
  // TMEM loads double-buffered: chunk c+1 is read while chunk c is stored
  uint32_t va[32], vb[32];
  __syncwarp();
  tmem_ld32(tbase + static_cast<uint32_t>(c0 * 32), va);
  tmem_ld_wait(va);
#pragma unroll
  for (int k = 0; k < kChunksPerWarp; ++k) {
    const int c = c0 + k;
    uint32_t(&cur_v)[32] = (k & 1) ? vb : va;
    uint32_t(&next_v)[32] = (k & 1) ? va : vb;
    if (k + 1 < kChunksPerWarp) {
      __syncwarp();
      tmem_ld32(tbase + static_cast<uint32_t>((c + 1) * 32), next_v);
    }
    bool staged = false;
    if (PHASE != 0) {
      staged = op.block(c) != nullptr;
      // this chunk's copies have landed (chunk c + 1's may still be in flight)
      if (k + 1 < kChunksPerWarp)
        fetch_wait<1>();
      else
        fetch_wait<0>();
    }
    epilogue_chunk<PHASE>(sc, ti, r, c, cur_v, staged, tiles[k & 1]);
    // the tile is free again (epilogue_chunk ends converged): chunk c + 2's operand into it
    if (PHASE != 0 && k + 2 < kChunksPerWarp) fetch_chunk(op, c + 2, tiles[k & 1]);
    if (k + 1 < kChunksPerWarp) {
      __syncwarp();
      tmem_ld_wait(next_v);
    }
  }
  return true;
}

// ---------------------------------------------------------------- fp32 path
// Each of the iterates, A and B is three bf16 slices (see part_a); the
// slices of one tensor are consecutive buffers, `slice` elements apart.
__device__ __forceinline__ size_t slice_m(const MatDesc &d) { return static_cast<size_t>(d.m) * d.pm; }
__device__ __forceinline__ size_t slice_s(const MatDesc &d) { return static_cast<size_t>(d.M) * d.ps; }

__device__ __forceinline__ float bf16_bits_to_float(uint32_t w, int hi) {
  return __uint_as_float(hi ? (w & 0xffff0000u) : (w << 16));
}

// Row `row` (< row_lim), columns col .. col+31 (zero at and past col_lim) of
// a sliced tensor, as the sum of its three slices (h + m first, then l).
__device__ __forceinline__ void sliced_row(const void *base_v, size_t slice, int pitch, int row, int row_lim,
                                           int col, int col_lim, float (&v)[32]) {
  const __nv_bfloat16 *base = static_cast<const __nv_bfloat16 *>(base_v);
  if (row >= row_lim) {
#pragma unroll
    for (int t = 0; t < 32; ++t) v[t] = 0.f;
    return;
  }
  const __nv_bfloat16 *p = base + static_cast<size_t>(row) * pitch + col;
  if (col + 32 <= col_lim) {  // 16-byte words: pitches are multiples of 8 elements, col of 32
    uint4 w[3][4];
#pragma unroll
    for (int z = 0; z < 3; ++z)
#pragma unroll
      for (int q = 0; q < 4; ++q) w[z][q] = __ldg(reinterpret_cast<const uint4 *>(p + z * slice) + q);
#pragma unroll
    for (int t = 0; t < 32; ++t) {
      float e[3];
#pragma unroll
      for (int z = 0; z < 3; ++z) {
        const uint4 &q = w[z][t >> 3];
        const int i = (t >> 1) & 3;
        e[z] = bf16_bits_to_float(i == 0 ? q.x : i == 1 ? q.y : i == 2 ? q.z : q.w, t & 1);
      }
      v[t] = (e[0] + e[1]) + e[2];
    }
  } else {
#pragma unroll
    for (int t = 0; t < 32; ++t)
      v[t] = col + t < col_lim ? (__bfloat162float(p[t]) + __bfloat162float(p[slice + t])) +
                                     __bfloat162float(p[2 * slice + t])
                               : 0.f;
  }
}

// Stores the 32 x 32 block v (one row per lane, rows row0.., columns col0..)
// as the three bf16 slices of a sliced tensor; v is consumed.
__device__ __forceinline__ void store_sliced(uint32_t *stage, float (&v)[32], void *base_v, size_t slice,
                                             size_t pitch, int row0, int row_lim, int col0, int col_lim,
                                             int *status) {
  __nv_bfloat16 *base = static_cast<__nv_bfloat16 *>(base_v);
  float g[32];
#pragma unroll
  for (int z = 0; z < 2; ++z) {
#pragma unroll
    for (int t = 0; t < 32; ++t) g[t] = __bfloat162float(__float2bfloat16_rn(v[t]));
    warp_store_rows(stage, g, base + z * slice, pitch, row0, row_lim, col0, col_lim, false, status);
#pragma unroll
    for (int t = 0; t < 32; ++t) v[t] -= g[t];  // exact: v and g agree in their leading bits
  }
  warp_store_rows(stage, v, base + 2 * slice, pitch, row0, row_lim, col0, col_lim, false, status);
}

// Word offset of 16-byte piece `piece` (0..7) of row `row` (0..31) in a
// 32 x 32 fp32 staging block (both staging tiles of a warp): the row-per-lane
// layout and the coalesced one (access k, lane l: piece l % 8 of row
// 4k + l / 8) are both bank-conflict free.
__device__ __forceinline__ int stage_word_f32(int row, int piece) { return row * 32 + 4 * (piece ^ (row & 7)); }

// As warp_store_rows for an fp32 destination (the caller's Y on the last
// step of the fp32 path): each store instruction writes 4 rows x 128 bytes.
__device__ __forceinline__ void warp_store_rows_f32(uint32_t *stage, const float (&v)[32], float *base, size_t pitch,
                                                    int row0, int row_lim, int col0, int col_lim, int *status) {
  const size_t bytes = static_cast<size_t>(row_lim) * pitch * 4;
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int q = 0; q < 8; ++q)
    *reinterpret_cast<uint4 *>(stage + stage_word_f32(lane, q)) =
        make_uint4(__float_as_uint(v[4 * q]), __float_as_uint(v[4 * q + 1]), __float_as_uint(v[4 * q + 2]),
                   __float_as_uint(v[4 * q + 3]));
  __syncwarp();
  const int piece = lane & 7;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int rl = 4 * k + (lane >> 3);
    const int R = row0 + rl, C0 = col0 + 4 * piece;
    if (R < row_lim && C0 < col_lim) {
      const uint4 o = *reinterpret_cast<const uint4 *>(stage + stage_word_f32(rl, piece));
      float *dst = base + static_cast<size_t>(R) * pitch + C0;
      if (C0 + 4 <= col_lim && (reinterpret_cast<uintptr_t>(dst) & 15) == 0) {
        if (in_bounds(dst, 16, base, bytes, status)) *reinterpret_cast<uint4 *>(dst) = o;
      } else {
        const uint32_t e[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (C0 + u < col_lim && in_bounds(dst + u, 4, base, bytes, status)) dst[u] = __uint_as_float(e[u]);
      }
    }
  }
  __syncwarp();
}

// Epilogue of one 32-column chunk on the fp32 path: as epilogue_chunk, with
// the re-read operand summed from its slices and the results stored as
// slices (fp32 into the caller's Y on the last step).
template <int PHASE>
__device__ __forceinline__ void epilogue_chunk_split(const StepCtx &p, const TileInfo &ti, int r, int chunk,
                                                     const uint32_t (&raw)[32], uint32_t *stage) {
  const MatDesc &d = *ti.d;
  const int r0 = r & ~31;
  float f[32];
#pragma unroll
  for (int t = 0; t < 32; ++t) f[t] = __uint_as_float(raw[t]);
  if (PHASE == 0 || PHASE == 1) {
    const int m = d.m, pm = d.pm;
    const int i = ti.row0 + r, i0 = ti.row0 + r0, jb = ti.col0 + chunk * 32;
    if (i0 >= m || jb >= m) return;  // warp-uniform
    if (PHASE == 0) {
#pragma unroll
      for (int t = 0; t < 32; ++t) f[t] *= p.gs;
    } else {
      float aold[32];
      sliced_row(d.a, slice_m(d), pm, i, m, jb, m, aold);
#pragma unroll
      for (int t = 0; t < 32; ++t) f[t] = p.cb * aold[t] + p.cc * f[t];
    }
    store_sliced(stage, f, PHASE == 0 ? d.a : d.b, slice_m(d), pm, i0, m, jb, m, p.status);
  } else {
    const int M = d.M, N = d.N;
    const int R = ti.row0 + r, R0 = ti.row0 + r0, C = ti.col0 + chunk * 32;
    if (R0 >= M || C >= N) return;  // warp-uniform
    float xo[32];
    sliced_row(d.s[p.step & 1], slice_s(d), d.ps, R, M, C, N, xo);
#pragma unroll
    for (int t = 0; t < 32; ++t) f[t] = p.as * (p.ca * xo[t] + f[t]);
    if (!p.final_step)
      store_sliced(stage, f, d.s[(p.step + 1) & 1], slice_s(d), static_cast<size_t>(d.ps), R0, M, C, N, p.status);
    else
      warp_store_rows_f32(stage, f, static_cast<float *>(d.user), static_cast<size_t>(N), R0, M, C, N, p.status);
  }
}

// Epilogue of one item on the fp32 path (its k-loop is six times as long,
// so the chunks are drained one TMEM load at a time).
template <int PHASE>
__device__ __forceinline__ bool epilogue_item_split(const StepCtx &sc, const TileInfo &ti, int r, int c0,
                                                    uint32_t tbase, uint32_t *stage, uint64_t *tfull, uint32_t parity,
                                                    const Waiter &w) {
  if (!mbar_wait<true>(tfull, parity, w)) return false;
  tc_fence_after();
  uint32_t v[32];
#pragma unroll 1
  for (int k = 0; k < kChunksPerWarp; ++k) {
    __syncwarp();
    tmem_ld32(tbase + static_cast<uint32_t>((c0 + k) * 32), v);
    tmem_ld_wait(v);
    epilogue_chunk_split<PHASE>(sc, ti, r, c0 + k, v, stage);
  }
  return true;
}

// A wait of a whole warp that only lane 0 polls (the other lanes sleep in
// the shuffle that broadcasts the outcome), leaving the warp converged.
template <bool kCluster>
__device__ __forceinline__ bool warp_mbar_wait(uint64_t *bar, uint32_t parity, const Waiter &w) {
  int ok = 1;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait<kCluster>(bar, parity, w) ? 1 : 0;
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// The producer's copies of one segment of an item in one CTA: for each
// k-block, wait for the stage to be free, and load this CTA's share of both
// operands (a0, b0: first tile row of each share) onto the leader's full
// barrier.
template <int AMN, int BMN, int kSplit = 0>
__device__ __forceinline__ bool produce_segment(int kb0, int kb1, const void *map_a, const void *map_b, int a0, int b0,
                                                uint8_t *sA, uint8_t *sB, Barriers *bar, bool leader, int &stage,
                                                uint32_t &phase_bit, int *issued_phase, uint64_t pol,
                                                const Waiter &w, int za = 0, int zb = 0) {
  for (int kb = kb0; kb < kb1; ++kb) {
    if (!warp_mbar_wait<true>(&bar->empty[stage], phase_bit ^ 1u, w)) return false;
    if (elect_one()) {
      if (leader) mbar_arrive_expect_tx(&bar->full[stage], kPairStageBytes);
      const uint32_t full_leader = mapa_shared(smem_u32(&bar->full[stage]), 0);
      const int kx = kb * kTcBK;
      load_operand<AMN, kSplit>(sA + stage * kABytes, map_a, a0, kx, za, full_leader, pol);
      load_operand<BMN, kSplit>(sB + stage * kBBytes, map_b, b0, kx, zb, full_leader, pol);
    }
    __syncwarp();
    issued_phase[stage] = static_cast<int>(phase_bit);
    if (++stage == kStages) {
      stage = 0;
      phase_bit ^= 1u;
    }
  }
  return true;
}

// The leader's MMAs of one segment of an item: for each k-block, wait for
// both CTAs' operand shares, issue the four K = 16 pair MMAs into `d_tmem`
// (accumulating from the item's first k-block of its first part on) and
// release the stage to both producers. AMN / BMN: MN-major first / second operand.
template <int AMN, int BMN>
__device__ __forceinline__ bool mma_segment(uint32_t d_tmem, int kb0, int kb1, uint8_t *sA, uint8_t *sB,
                                            Barriers *bar, int &stage, uint32_t &phase_bit, const Waiter &w,
                                            int part = 0) {
  constexpr uint32_t idesc = umma_idesc_bf16(kTcCluster * kTcBM, kTcBN, AMN, BMN);
  constexpr uint16_t kPairMask = (1u << kTcCluster) - 1;
  for (int kb = kb0; kb < kb1; ++kb) {
    if (!warp_mbar_wait<true>(&bar->full[stage], phase_bit, w)) return false;
    tc_fence_after();
    const uint32_t a_addr = smem_u32(sA + stage * kABytes);
    const uint32_t b_addr = smem_u32(sB + stage * kBBytes);
    if (elect_one()) {
#pragma unroll
      for (int k = 0; k < kTcBK / 16; ++k)
        umma_bf16_pair(d_tmem, operand_desc<AMN>(a_addr, k), operand_desc<BMN>(b_addr, k), idesc,
                       (part | kb | k) != 0 ? 1u : 0u);
      umma_commit_pair_multicast(&bar->empty[stage], kPairMask);
    }
    __syncwarp();
    if (++stage == kStages) {
      stage = 0;
      phase_bit ^= 1u;
    }
  }
  return true;
}

// kQueued: the pair's items come from the leader's fetcher through the
// shared-memory queue (tickets or stride; the single-launch schedule);
// otherwise every role walks the pair's static stride itself (per-phase
// launches), which keeps that kernel's code and registers to what it needs.
// kSplit: the fp32 path (per-phase launches only), every tensor three bf16
// slices and every item six slice products (see part_a).
template <bool kQueued, int kSplit = 0>
__global__ void __launch_bounds__(kThreads, 1) ns_tc_gemm_kernel(const __grid_constant__ TcParams p) {
  static_assert(!(kQueued && kSplit), "the fp32 path runs per-phase launches");
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *sA = smem;
  uint8_t *sB = smem + kStages * kABytes;
  Barriers *bar = reinterpret_cast<Barriers *>(smem + kStages * kStageBytes);
  uint32_t *epi_stage = reinterpret_cast<uint32_t *>(smem + kStages * kStageBytes + kBarrierBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int cluster = blockIdx.x / kTcCluster;
  const int nclusters = gridDim.x / kTcCluster;
  const int my_rows = static_cast<int>(rank) * kTcBM;
  constexpr uint16_t kPairMask = (1u << kTcCluster) - 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bar->full[s], 1);
      mbar_init(&bar->empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&bar->tfull[a], 1);
      mbar_init(&bar->tempty[a], kTcCluster * kEpiWarps);  // one arrival per epilogue warp
      mbar_init(&bar->epi_done[a], kEpiWarps);
    }
    for (int q = 0; q < kQueue; ++q) {
      mbar_init(&bar->qfull[q], 1);
      mbar_init(&bar->qempty[q], kQueueConsumers);
    }
    mbar_init(&bar->drain, 1);
    bar->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(&bar->tmem_base, kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = bar->tmem_base;
  // the pair MMA writes the same TMEM columns in both CTAs: check that both
  // allocations agree before using them
  const uint32_t peer_tmem = ld_shared_cluster_u32(mapa_shared(smem_u32(&bar->tmem_base), rank ^ 1u));
  const bool tmem_ok = peer_tmem == tmem;
  if (!tmem_ok && threadIdx.x == 0) set_status(p.status, kStatusTmemMismatch);
  volatile int *abort = &bar->abort;
  const Waiter w{abort, p.status, p.wait_limit_ns};

  if constexpr (kQueued) {
  if (tmem_ok && warp == 0) {
    {
      // ---------------------------------------------------- TMA producer (both CTAs)
      // the whole warp runs the loop; one elected lane issues each copy. In
      // the leader this warp is also the pair's fetcher: it takes the pair's
      // items (tickets or static stride) and publishes them to both queues.
      const uint64_t pol = l2_policy_evict_normal();
      int issued_phase[kStages];
      for (int s = 0; s < kStages; ++s) issued_phase[s] = -1;
      int stage = 0;
      uint32_t phase_bit = 0;
      bool ok = true;
      // The fetcher publishes every item one item ahead of its own production
      // of it, so the peer's producer and the other roles have each item a
      // whole tile before they need it.
      Fetcher f;
      QItem next;
      next.g = p.g_end;
      if (leader) {
        fetcher_start(p, p.g_begin + cluster, nclusters, f);
        next = fetcher_item(f);
        int put = 1;
        if (lane == 0) put = queue_put(bar, 0, next, w) ? 1 : 0;
        ok = __shfl_sync(0xffffffffu, put, 0) != 0;
        if (ok && next.g < p.g_end) fetcher_advance(p, nclusters, f);
      }
      for (int k = 0; ok; ++k) {
        QItem it;
        if (leader) {
          it = next;
          if (it.g >= p.g_end) break;
          // publish item k + 1 now; the lookups of the items after it run
          // while item k is produced
          next = fetcher_item(f);
          int put = 1;
          if (lane == 0) put = queue_put(bar, k + 1, next, w) ? 1 : 0;
          if (!__shfl_sync(0xffffffffu, put, 0)) break;
          if (next.g < p.g_end) {
            fetcher_advance(p, nclusters, f);
            if (f.g < p.g_end && elect_one()) prefetch_item_maps(p.mats[f.tl.mat], f.sp >> 4, (f.sp >> 2) & 3);
            __syncwarp();
          }
        } else if (!queue_get_warp(bar, k, it, w)) {
          break;
        }
        if (it.g >= p.g_end) break;
        const TileInfo ti = item_info(p, it);
        if (ti.skip) continue;
        if (p.wait) {
          // operands come from earlier phases of this matrix, written by
          // epilogues anywhere on the GPU
          int ready = 1;
          if (lane == 0) ready = wait_count(p.done + ti.mat, units_before(*ti.d, it.step(), it.phase()), w) ? 1 : 0;
          if (!__shfl_sync(0xffffffffu, ready, 0)) break;
          fence_proxy_async_global();
        }
        const ItemPlan pl = plan_item(*ti.d, it.step(), it.phase(), ti.tr, it.direct(), ti.row0, ti.col0, ti.nk);
        const int a0 = ti.row0 + my_rows, b0 = ti.col0 + static_cast<int>(rank) * (kTcBN / 2);
        // one k-loop per operand order, so the copies issued are exactly the ones needed
        ok = produce_segment<1, 1>(0, pl.e0, pl.map[0][0], pl.map[0][1], a0, b0, sA, sB, bar, leader, stage,
                                   phase_bit, issued_phase, pol, w);
        if (ok)
          ok = produce_segment<0, 1>(pl.e0, pl.e1, pl.map[1][0], pl.map[1][1], a0, b0, sA, sB, bar, leader, stage,
                                     phase_bit, issued_phase, pol, w);
        if (ok)
          ok = produce_segment<0, 0>(pl.e1, ti.nk, pl.map[2][0], pl.map[2][1], a0, b0, sA, sB, bar, leader, stage,
                                     phase_bit, issued_phase, pol, w);
      }
      if (*abort && leader && lane == 0) {
        for (int s = 0; s < kStages; ++s)
          if (issued_phase[s] >= 0) mbar_drain(&bar->full[s], static_cast<uint32_t>(issued_phase[s]), w);
      }
    }
  } else if (tmem_ok && warp == 1) {
    if (leader) {
      // ---------------------------------------------------- pair MMA issuer (leader)
      // the whole warp runs the loop; one elected lane issues the MMAs and commits
      int stage = 0;
      uint32_t phase_bit = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      // items are read from the queue one item ahead (each is published
      // before the item in front of it is produced), so the step from one
      // item's last MMAs to the next item's first costs no queue access
      QItem nxt;
      bool have = queue_get_warp(bar, 0, nxt, w);
      for (int k = 0; ok && have; ++k) {
        const QItem it = nxt;
        if (it.g >= p.g_end) break;
        have = queue_get_warp(bar, k + 1, nxt, w);
        const TileInfo ti = item_info(p, it);
        if (ti.skip) continue;
        const ItemPlan pl = plan_item(*ti.d, it.step(), it.phase(), ti.tr, it.direct(), ti.row0, ti.col0, ti.nk);
        if (!warp_mbar_wait<true>(&bar->tempty[acc], acc_phase ^ 1u, w)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem + static_cast<uint32_t>(acc * kTcBN);
        // one k-loop per operand order, so descriptors stay compile-time
        ok = mma_segment<1, 1>(d_tmem, 0, pl.e0, sA, sB, bar, stage, phase_bit, w);
        if (ok) ok = mma_segment<0, 1>(d_tmem, pl.e0, pl.e1, sA, sB, bar, stage, phase_bit, w);
        if (ok) ok = mma_segment<0, 0>(d_tmem, pl.e1, ti.nk, sA, sB, bar, stage, phase_bit, w);
        if (!ok) break;
        if (elect_one()) umma_commit_pair_multicast(&bar->tfull[acc], kPairMask);
        __syncwarp();
        if (++acc == kAccs) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      if (elect_one()) {
        umma_commit_pair_multicast(&bar->drain, 1u);
        mbar_drain(&bar->drain, 0, w);
      }
      __syncwarp();
    }
  } else if (tmem_ok && warp < kSignalWarp) {
    // ------------------------------------------------------ epilogue (both CTAs)
    // warps 2..9: TMEM lane quarter q = warp % 4 (tile rows q*32 .. q*32+31),
    // column half h: chunks h*kChunksPerWarp .. of the 256 accumulator columns
    const int e = warp - 2;
    const int q = warp & 3;
    const int r = q * 32 + lane;
    const int c0 = (e / 4) * kChunksPerWarp;
    uint32_t *stage = epi_stage + e * (kEpiStageBytes / 4);
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int k = 0;; ++k) {
      QItem it;
      if (!queue_get_warp(bar, k, it, w) || it.g >= p.g_end) break;
      TileInfo ti = item_info(p, it);
      if (ti.skip) continue;
      if (p.wait) {
        // the operand this epilogue reloads (A, or the current iterate) comes from an earlier phase
        bool ready = true;
        if (lane == 0) ready = wait_count(p.done + ti.mat, units_before(*ti.d, it.step(), it.phase()), w);
        if (!__shfl_sync(0xffffffffu, ready ? 1 : 0, 0)) break;
        __syncwarp();  // orders the other lanes' reads after lane 0's acquire
      }
      ti.row0 += my_rows;
      const StepCtx sc = step_ctx(p, it.step(), ti.mat);
      const uint32_t tbase = tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * kTcBN);
      bool ok;
      const int phase = it.phase();
      if (phase == 0)
        ok = epilogue_item<0>(sc, ti, r, c0, tbase, stage, &bar->tfull[acc], acc_phase, w);
      else if (phase == 1)
        ok = epilogue_item<1>(sc, ti, r, c0, tbase, stage, &bar->tfull[acc], acc_phase, w);
      else
        ok = epilogue_item<2>(sc, ti, r, c0, tbase, stage, &bar->tfull[acc], acc_phase, w);
      if (!ok) break;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive_cluster(mapa_shared(smem_u32(&bar->tempty[acc]), 0));  // TMEM reusable
        mbar_arrive(&bar->epi_done[acc]);                                   // stores issued (release)
      }
      if (++acc == kAccs) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  } else if (tmem_ok && warp == kSignalWarp) {
    if (lane == 0) {
      // ---------------------------------------------------- completion signal (both CTAs)
      // After the CTA's epilogue warps stored an item (their arrivals on
      // epi_done release the stores to this thread), publish it at GPU scope;
      // the release is cumulative, so a consumer that acquires the counter
      // sees every store of the item. Skipped items are published once their
      // own dependencies are met.
      int acc = 0;
      uint32_t acc_phase = 0;
      for (int k = 0;; ++k) {
        QItem it;
        if (!queue_get_lane(bar, k, it, w)) break;
        const TileInfo ti = item_info(p, it);
        queue_release(bar, k);  // after the item was used
        if (it.g >= p.g_end) break;
        if (ti.skip) {
          if (p.wait && !wait_count(p.done + ti.mat, units_before(*ti.d, it.step(), it.phase()), w)) break;
        } else {
          if (!mbar_wait(&bar->epi_done[acc], acc_phase, w)) break;
          if (++acc == kAccs) {
            acc = 0;
            acc_phase ^= 1u;
          }
        }
        if (!p.hold_signals) red_release_gpu_add(p.done + ti.mat, 1);
      }
    }
  }

  } else {
  if (tmem_ok && warp == 0) {
    {
      // ---------------------------------------------------- TMA producer (both CTAs)
      // the whole warp runs the loop; one elected lane issues each copy
      const uint64_t pol = l2_policy_evict_normal();
      int issued_phase[kStages];
      for (int s = 0; s < kStages; ++s) issued_phase[s] = -1;
      int stage = 0;
      uint32_t phase_bit = 0;
      bool ok = true;
      ItemPipe q;
      pipe_start(p, p.g_begin + cluster, nclusters, q);
      while (q.g < p.g_end && ok) {
        int step, phase, direct;
        TileInfo ti;
        pipe_take(p, nclusters, q, step, phase, ti, direct);
        if (q.g < p.g_end && elect_one()) prefetch_item_maps_exact(p.mats[q.tl.mat], q.step, q.phase, q.tr, q.direct);
        __syncwarp();
        if (ti.skip) continue;
        if (p.wait) {
          // operands come from earlier phases of this matrix, written by
          // epilogues anywhere on the GPU
          int ready = 1;
          if (lane == 0) ready = wait_count(p.done + ti.mat, units_before(*ti.d, step, phase), w) ? 1 : 0;
          if (!__shfl_sync(0xffffffffu, ready, 0)) break;
          fence_proxy_async_global();
        }
        const ItemPlan pl = plan_item(*ti.d, step, phase, ti.tr, direct, ti.row0, ti.col0, ti.nk);
        const int a0 = ti.row0 + my_rows, b0 = ti.col0 + static_cast<int>(rank) * (kTcBN / 2);
        // one k-loop per operand order, so the copies issued are exactly the ones needed
        // (per slice product on the fp32 path)
        for (int part = 0; ok && part < (kSplit ? kSplitParts : 1); ++part) {
          const int za = kSplit ? part_a(part) : 0, zb = kSplit ? part_b(part) : 0;
          ok = produce_segment<1, 1, kSplit>(0, pl.e0, pl.map[0][0], pl.map[0][1], a0, b0, sA, sB, bar, leader, stage,
                                             phase_bit, issued_phase, pol, w, za, zb);
          if (ok)
            ok = produce_segment<0, 1, kSplit>(pl.e0, pl.e1, pl.map[1][0], pl.map[1][1], a0, b0, sA, sB, bar, leader,
                                               stage, phase_bit, issued_phase, pol, w, za, zb);
          if (ok)
            ok = produce_segment<0, 0, kSplit>(pl.e1, ti.nk, pl.map[2][0], pl.map[2][1], a0, b0, sA, sB, bar, leader,
                                               stage, phase_bit, issued_phase, pol, w, za, zb);
        }
      }
      if (*abort && leader && lane == 0) {
        for (int s = 0; s < kStages; ++s)
          if (issued_phase[s] >= 0) mbar_drain(&bar->full[s], static_cast<uint32_t>(issued_phase[s]), w);
      }
    }
  } else if (tmem_ok && warp == 1) {
    if (leader) {
      // ---------------------------------------------------- pair MMA issuer (leader)
      // the whole warp runs the loop; one elected lane issues the MMAs and commits
      int stage = 0;
      uint32_t phase_bit = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      ItemPipe q;
      pipe_start(p, p.g_begin + cluster, nclusters, q);
      while (q.g < p.g_end && ok) {
        int step, phase, direct;
        TileInfo ti;
        pipe_take(p, nclusters, q, step, phase, ti, direct);
        if (ti.skip) continue;
        const ItemPlan pl = plan_item(*ti.d, step, phase, ti.tr, direct, ti.row0, ti.col0, ti.nk);
        if (!warp_mbar_wait<true>(&bar->tempty[acc], acc_phase ^ 1u, w)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem + static_cast<uint32_t>(acc * kTcBN);
        // one k-loop per operand order, so descriptors stay compile-time
        // (per slice product on the fp32 path)
        for (int part = 0; ok && part < (kSplit ? kSplitParts : 1); ++part) {
          ok = mma_segment<1, 1>(d_tmem, 0, pl.e0, sA, sB, bar, stage, phase_bit, w, part);
          if (ok) ok = mma_segment<0, 1>(d_tmem, pl.e0, pl.e1, sA, sB, bar, stage, phase_bit, w, part);
          if (ok) ok = mma_segment<0, 0>(d_tmem, pl.e1, ti.nk, sA, sB, bar, stage, phase_bit, w, part);
        }
        if (!ok) break;
        if (elect_one()) umma_commit_pair_multicast(&bar->tfull[acc], kPairMask);
        __syncwarp();
        if (++acc == kAccs) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      if (elect_one()) {
        umma_commit_pair_multicast(&bar->drain, 1u);
        mbar_drain(&bar->drain, 0, w);
      }
      __syncwarp();
    }
  } else if (tmem_ok && warp < kSignalWarp) {
    // ------------------------------------------------------ epilogue (both CTAs)
    // warps 2..9: TMEM lane quarter q = warp % 4 (tile rows q*32 .. q*32+31),
    // column half h: chunks h*kChunksPerWarp .. of the 256 accumulator columns
    const int e = warp - 2;
    const int q = warp & 3;
    const int r = q * 32 + lane;
    const int c0 = (e / 4) * kChunksPerWarp;
    uint32_t *stage = epi_stage + e * (kEpiStageBytes / 4);
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int g = p.g_begin + cluster; g < p.g_end; g += nclusters) {
      int step, phase, t;
      decode_item(p, g, step, phase, t);
      TileInfo ti = tile_info(p, phase, t);
      if (ti.skip) continue;
      if (p.wait) {
        // the operand this epilogue reloads (A, or the current iterate) comes from an earlier phase
        bool ready = true;
        if (lane == 0) ready = wait_count(p.done + ti.mat, units_before(*ti.d, step, phase), w);
        if (!__shfl_sync(0xffffffffu, ready ? 1 : 0, 0)) break;
      }
      ti.row0 += my_rows;
      const StepCtx sc = step_ctx(p, step, ti.mat);
      const uint32_t tbase = tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * kTcBN);
      bool ok;
      if constexpr (kSplit) {
        if (phase == 0)
          ok = epilogue_item_split<0>(sc, ti, r, c0, tbase, stage, &bar->tfull[acc], acc_phase, w);
        else if (phase == 1)
          ok = epilogue_item_split<1>(sc, ti, r, c0, tbase, stage, &bar->tfull[acc], acc_phase, w);
        else
          ok = epilogue_item_split<2>(sc, ti, r, c0, tbase, stage, &bar->tfull[acc], acc_phase, w);
      } else {
        if (phase == 0)
          ok = epilogue_item<0>(sc, ti, r, c0, tbase, stage, &bar->tfull[acc], acc_phase, w);
        else if (phase == 1)
          ok = epilogue_item<1>(sc, ti, r, c0, tbase, stage, &bar->tfull[acc], acc_phase, w);
        else
          ok = epilogue_item<2>(sc, ti, r, c0, tbase, stage, &bar->tfull[acc], acc_phase, w);
      }
      if (!ok) break;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive_cluster(mapa_shared(smem_u32(&bar->tempty[acc]), 0));  // TMEM reusable
        mbar_arrive(&bar->epi_done[acc]);                                   // stores issued (release)
      }
      if (++acc == kAccs) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  } else if (tmem_ok && warp == kSignalWarp) {
    if (lane == 0) {
      // ---------------------------------------------------- completion signal (both CTAs)
      // After the CTA's epilogue warps stored an item (their arrivals on
      // epi_done release the stores to this thread), publish it at GPU scope;
      // the release is cumulative, so a consumer that acquires the counter
      // sees every store of the item. Skipped items are published once their
      // own dependencies are met.
      int acc = 0;
      uint32_t acc_phase = 0;
      for (int g = p.g_begin + cluster; g < p.g_end; g += nclusters) {
        int step, phase, t;
        decode_item(p, g, step, phase, t);
        const TileInfo ti = tile_info(p, phase, t);
        if (ti.skip) {
          if (p.wait && !wait_count(p.done + ti.mat, units_before(*ti.d, step, phase), w)) break;
        } else {
          if (!mbar_wait(&bar->epi_done[acc], acc_phase, w)) break;
          if (++acc == kAccs) {
            acc = 0;
            acc_phase ^= 1u;
          }
        }
        if (!p.hold_signals) red_release_gpu_add(p.done + ti.mat, 1);
      }
    }
  }

  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem, kTmemCols);
}

int launch_tc_kernel(const TcParams &p, int max_ctas, cudaStream_t s) {
  const int smem = tc_smem_bytes();
  const int variant = p.tickets ? 1 : (p.split ? 2 : 0);
  auto kernel = variant == 1 ? ns_tc_gemm_kernel<true> : (variant == 2 ? ns_tc_gemm_kernel<false, 1> : ns_tc_gemm_kernel<false>);
  static SmemOptIn opt_in[3];
  if (opt_in[variant].ensure(reinterpret_cast<const void *>(kernel), smem)) return -1;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kTcCluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // items that wait on other clusters' items need every CTA resident at once
  attr[1].id = cudaLaunchAttributeCooperative;
  attr[1].val.cooperative = 1;
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // persistent: as many pairs as can be resident at once (items wait on one
  // another, so every pair of the grid must be resident), at most one per item
  static int resident_pairs[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  int &cached = resident_pairs[dev & 63];
  if (cached == 0) {
    cfg.gridDim = dim3(kTcCluster * (max_ctas / kTcCluster), 1, 1);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      return -1;
    }
    cached = n;
  }
  const int items = p.g_end - p.g_begin;
  const int pairs = cached < items ? cached : items;
  cfg.gridDim = dim3(kTcCluster * pairs, 1, 1);
  cfg.numAttrs = p.wait ? 2 : 1;
  if (cudaLaunchKernelEx(&cfg, kernel, p) != cudaSuccess) {
    cudaGetLastError();
    return p.wait ? 1 : -1;  // 1: a co-resident launch was refused; the caller can split by phase
  }
  count_launch();
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace

static_assert(1024 + kStages * kStageBytes + kBarrierBytes + kEpiWarps * kEpiStageBytes <= 227 * 1024,
              "shared memory of the tensor-core kernel");

int tc_smem_bytes() { return 1024 + kStages * kStageBytes + kBarrierBytes + kEpiWarps * kEpiStageBytes; }

int launch_tc(const TcParams &p, int max_ctas, cudaStream_t s) {
  if (p.g_end <= p.g_begin) return 0;
  return launch_tc_kernel(p, max_ctas, s);
}

}  // namespace ns
