// moe_fp8_block_scale_forward: the fused block-scaled FP8 MoE expert
// computation on GB300 (FlashInfer PR #4287: commit summary; "Public contract
// and review fixes"; post-dot scale application from "Final W8 kernel
// performance (v46)").
//
// Launches on the caller's stream:
//   0. stage: per plan slot, the route's token and weight and the activation
//      block scales (transposed, one row per K slice); per (plan block,
//      n tile, K slice) a 16-byte record of the two weight block scales the
//      tile needs; for well-filled plans also the activation rows themselves,
//      in plan order.  Everything the GEMM epilogues need thus arrives by TMA.
//   1. up   (gemm kernel, kUp = true): for every (plan block, 256-wide tile of
//      the interleaved gate/up weights): activation rows x W13 tile on
//      tcgen05 tensor cores, one 128-wide K slice at a time into TMEM; the
//      epilogue warps promote each slice in FP32 with the activation and
//      weight block scales, then apply SwiGLU and requantise the 128
//      intermediate columns of the tile to E4M3 (scale amax/448) into the
//      workspace (the codes leave through tensor stores of row boxes).
//   2. down (gemm kernel, kUp = false): intermediate rows x W2 tile, promoted
//      with the intermediate and W2 block scales, times the route weight and
//      routed scale, rounded to BF16 and stored as the route's row of the
//      workspace (row index = route id).
//   3. combine: out = bf16_rn(f32(out) + sum of the token's route rows).
// Sparse plans (decode) take the vector path instead (vector.cu).
//
// The GEMM kernel is persistent and warp specialised (320 threads):
//   warp 0      TMA producer: activation (or intermediate) rows, the 256-row
//               weight tile and the slice's scales into a 4-stage ring;
//   warp 1      TMEM allocation and the single MMA-issuing thread
//               (kind::f8f6f4, M=128, N=256, K=32 per instruction, 4 per slice);
//   warps 2..9  epilogue: each owns 32 tile rows (its TMEM lane quarter) and
//               128 of the 256 columns; FP32 accumulators live in registers.
// TMEM holds two 256-column FP32 partial buffers so the tensor core computes
// slice k+1 while the epilogue promotes slice k.  A stage is refilled only
// after the MMA has consumed it and every epilogue warp has read its scales.
// The epilogue issues no global loads: under the weight stream a plain load
// waits behind the TMA traffic for several microseconds.
// Every wait is bounded; a wait that runs out raises MOE_DEV_TIMEOUT in
// *device_status and the CTA winds down (draining its copies and MMAs,
// freeing TMEM).
#include <mutex>

#include "common.cuh"
#include "vector.cuh"

namespace moe {
namespace {

constexpr int kTileM = 128;
constexpr int kTileN = 256;
constexpr int kTileK = 128;
constexpr int kABytes = kTileM * kTileK;  // 16 KiB
constexpr int kBBytes = kTileN * kTileK;  // 32 KiB
constexpr int kNumEpiWarps = 8;
constexpr int kNumThreads = 64 + 32 * kNumEpiWarps;
constexpr uint32_t kTmemCols = 512;
constexpr int kMaxStages = 5;
constexpr int kMaxBlocksSmem = 1024;  // plan blocks whose expert id is cached in shared memory
constexpr int kRowPad = kTileM;       // staged per-slot arrays carry this many extra slots

// Single CTA: 4 stages of 16 KiB activation rows + the 32 KiB weight tile.
// CTA pair (cta_group::2, M = 256 over two plan blocks of one expert): each
// CTA holds its own 128 rows and half (128 rows) of the weight tile, so a
// stage is 32 KiB and 5 stages fit.
template <bool kPair> struct Cfg {
  static constexpr int kStages = kPair ? 5 : 4;
  static constexpr int kBStage = kPair ? kBBytes / 2 : kBBytes;
  static constexpr uint32_t kIdesc = idesc_e4m3_f32(kPair ? 2 * kTileM : kTileM, kTileN);
};

// Per-stage side data, filled by bulk copies next to the operand tiles.
struct StageExtra {
  float a_scale[kTileM];     // activation (up) / intermediate (down) scale of each tile row
  int32_t tok[kTileM];       // first slice of a tile: route id of each row (-1 = no route)
  float weight[kTileM];      // down, first slice of a tile: route weight x routed scale
  float4 w_scale;            // the tile's two weight block scales for this K slice
  float4 pad0;
};
static_assert(sizeof(StageExtra) == 1568 && sizeof(StageExtra) % 16 == 0, "stage extra layout");

struct SmemCtl {
  uint64_t full[kMaxStages];       // operand tiles landed (the leader's counts both CTAs of a pair)
  uint64_t xfull[kMaxStages];      // this CTA's stage extras landed
  uint64_t empty[kMaxStages];      // stage free: MMA done + every local epilogue warp read its extras
  uint64_t tfull[2];
  uint64_t tempty[2];              // (leader) TMEM buffer released by every epilogue warp of the pair
  uint32_t tmem_base;
  int abort_flag;
  int last_flag;                   // split-K: this CTA completed the tile's sum
  int pad;
  union alignas(128) Scratch {  // (tensor stores read 128-byte aligned shared memory)
    struct {
      float xchg[2][2][kTileM];                 // [tile parity][column half][row] amax exchange
      // block-scaled mode: per stage, the slice's UE8M0 scale-factor rows
      // for the tensor-memory copy (A: 32 rows x 16 bytes, then B)
      alignas(16) uint8_t sf[kMaxStages][1024];
      // per epilogue warp, the codes of its 32 rows x 32 columns on their way
      // to q_inter through tensor stores
      alignas(128) uint8_t qst[kNumEpiWarps][32 * 32];
    } up;
    uint32_t yt[kNumEpiWarps][32][20];          // down: per-warp transpose of 32 rows x 32 BF16 (padded rows)
  } u;
  int32_t row_tok[kTileM];         // up with split K: token of each tile row (-1 = no route)
  int32_t expert[kMaxBlocksSmem];  // expert of each plan block (cached at start)
  uint8_t pairf[kMaxBlocksSmem];   // pair mode: bit 0 leads a pair, bit 1 has a partner
};

static_assert(offsetof(SmemCtl, u) % 16 == 0, "scratch alignment");
static_assert(sizeof(SmemCtl) % 16 == 0, "control block size");

static_assert(alignof(SmemCtl) == 128 && offsetof(SmemCtl, u) % 128 == 0, "control block alignment");

// 1024 bytes for aligning the operand stages, 128 for aligning the control block.
template <bool kPair>
constexpr size_t smem_bytes() {
  return 1024 + static_cast<size_t>(Cfg<kPair>::kStages) * (kABytes + Cfg<kPair>::kBStage + sizeof(StageExtra)) +
         128 + sizeof(SmemCtl);
}
static_assert(smem_bytes<false>() <= 232448 && smem_bytes<true>() <= 232448, "shared memory budget");

// Tensor-memory columns of the block-scaled mode: the accumulator (one
// 256-column buffer: a tile accumulates over all its K slices), then per
// stage 16 columns of scale factors (A at +0..3, B at +4..11).
constexpr uint32_t kSfTmemCol = kTileN;
constexpr uint32_t kIdescMx = idesc_mx_e4m3(kTileM, kTileN);

// A UE8M0 scale must be +0 or a normal power of two (exponent field 1..254,
// zero mantissa, positive).
__device__ __forceinline__ bool ue8m0_ok(float v) {
  const uint32_t bits = __float_as_uint(v);
  return bits == 0u || ((bits & 0x807FFFFFu) == 0u && (bits >> 23) != 0xFFu);
}
// The exponent byte of a power-of-two FP32 scale (0 for +0, i.e. 2^-127),
// in all four bytes of a tensor-memory cell.
__device__ __forceinline__ uint32_t ue8m0_word(float v) {
  return ((__float_as_uint(v) >> 23) & 0xFFu) * 0x01010101u;
}

struct GemmParams {
  const int32_t* expert_ids;
  const int32_t* num_post_padded;
  const int32_t* sorted_ids;   // up with gather4: plan (token of each row)
  const float* a_scale_t;      // [nkb, cap_pad]: scale of each plan slot per K slice
  const float4* w_scale_st;    // [nblocks, ntiles_n, nkb]: weight scales per tile and slice
  const int32_t* slot_route;   // [cap_pad] route id r = t * top_k + j per plan slot (-1 = pad)
  const float* slot_w;         // [cap_pad] route weight x routed scale
  uint16_t* y_out;             // down: [R, H] BF16 route contributions y * w, by route id
  uint8_t* q_inter;            // up: [sorted_cap, I]
  float* s_inter_t;            // up: [I/128, cap_pad]
  uint8_t* dbg_q;              // up, nullable: [sorted_cap, I]
  float* dbg_s;                // up, nullable: [sorted_cap, I/128]
  int32_t* status;             // nullable
  int64_t nblocks;             // plan block slots the grid walks
  int64_t cap_pad;             // row stride of the staged per-slot arrays
  int R;
  int top_k;
  int block_m;
  int E;
  int nkb;                     // K / 128
  int ntiles_n;                // 256-wide output tiles per expert
  int b_rows;                  // weight rows per expert (2I or H)
  int I;
  int H;
  int a_gather4;               // up only: 1 = activation rows fetched by token with tile::gather4,
                               //          0 = rows already in plan order (2D boxes by plan slot)
  int tile_group;              // tile order: 0 = all n tiles of a plan block together (block major);
                               // G > 0 = groups of G n tiles, within a group block major
  int splits;                  // up only: K splits per tile (1 = none)
  int ksplit;                  // K slices per split
  float* usum;                 // up, splits > 1: [nblocks, ntiles_n, block_m, 256] zeroed partial sums
  int32_t* ucnt;               // up, splits > 1: [nblocks, ntiles_n] zeroed arrival tickets
  uint32_t* gen;               // up: forward stamp, advanced once per forward
  int64_t a_rows;              // rows of the A operand's tensor (M tokens, or sorted_cap plan slots)
  int64_t q_rows;              // up: rows of q_inter (sorted_cap)
  int qbox;                    // up: rows per tensor store of codes (8, 16 or 32; divides block_m)
};

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          unsigned long long limit_ns = kWaitLimitNs) {
  int ok = 0;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, abort_flag, limit_ns) ? 1 : 0;
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// Bounded wait used while winding down: ignores the abort flag.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  int dummy = 0;
  mbar_wait(bar, parity, &dummy);
}

__device__ __forceinline__ void report(int32_t* status, int bits) {
  if (status) atomicOr(status, bits);
}

__device__ __forceinline__ int block_expert(const GemmParams& p, const SmemCtl* ctl, int64_t b) {
  if (b < kMaxBlocksSmem) return ctl->expert[b];
  return MOE_IN_BOUNDS(b < p.nblocks) ? p.expert_ids[b] : -1;
}

// Tile -> (plan block, n tile, K split, expert); false if the tile has no
// work.  In pair mode only blocks that lead a pair carry tiles.
template <bool kPair>
__device__ __forceinline__ bool tile_coords(const GemmParams& p, const SmemCtl* ctl, int64_t tile, int64_t nvalid,
                                            int& b, int& t, int& sp, int& e) {
  sp = static_cast<int>(tile % p.splits);
  const int64_t bt = tile / p.splits;
  if (p.tile_group == 0) {
    b = static_cast<int>(bt / p.ntiles_n);
    t = static_cast<int>(bt % p.ntiles_n);
  } else {
    const int64_t per_group = p.nblocks * p.tile_group;
    const int64_t g = bt / per_group, r = bt - g * per_group;
    b = static_cast<int>(r / p.tile_group);
    t = static_cast<int>(g * p.tile_group + r % p.tile_group);
  }
  if (b >= nvalid) return false;
  if (kPair && !(ctl->pairf[b] & 1)) return false;
  e = block_expert(p, ctl, b);
  return e >= 0 && e < p.E;
}

// Plan entries of the four rows 4*lane .. 4*lane+3 of plan block b (gather4 path).
__device__ __forceinline__ void load_ids(const GemmParams& p, int b, int lane, int (&id)[4]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = 4 * lane + i;
    const int64_t q = static_cast<int64_t>(b) * p.block_m + r;
    id[i] = (r < p.block_m && MOE_IN_BOUNDS(q < p.nblocks * p.block_m)) ? p.sorted_ids[q] : -1;
  }
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Arrive on an mbarrier of another CTA of the cluster.  Release at CTA scope
// is enough for its one use (handing a TMEM buffer back after the reads have
// completed); a cluster-scope release waits for the CTA's outstanding memory
// traffic and costs microseconds under the operand stream.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
// 2D tensor load whose completion is signalled on an mbarrier that may sit in
// the peer CTA of the pair (cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], "
      "[%2];" ::"r"(dst),
      "l"(map), "r"(bar), "r"(x), "r"(y)
      : "memory");
}

template <bool kPair>
__device__ __forceinline__ void tmem_alloc_k(uint32_t dst, uint32_t ncols) {
  if (kPair)
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst), "r"(ncols) : "memory");
  else
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst), "r"(ncols) : "memory");
}
template <bool kPair>
__device__ __forceinline__ void tmem_relinquish_k() {
  if (kPair)
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  else
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
template <bool kPair>
__device__ __forceinline__ void tmem_dealloc_k(uint32_t taddr, uint32_t ncols) {
  if (kPair)
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
  else
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// The MMA of the pair: M = 256 (128 rows in each CTA), B split along N.
__device__ __forceinline__ void umma_f8_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive on the same mbarrier in both CTAs of the pair once every MMA issued
// so far has completed.
__device__ __forceinline__ void umma_commit_pair(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
      "h"(static_cast<uint16_t>(3))
      : "memory");
}

// kBS (gate/up, single CTAs only): both operands' scales are powers of two,
// applied by the tensor core (kind::mxf8f6f4.block_scale) as UE8M0 scale
// factors; a tile accumulates over all its K slices in tensor memory and the
// epilogue reads it once, with no per-slice promotion.
template <bool kUp, bool kPair, bool kBS = false>
__global__ void __launch_bounds__(kNumThreads, 1)
    moe_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmQ, const GemmParams p) {
  static_assert(!kBS || (kUp && !kPair), "block-scaled mode: gate/up on single CTAs");
  using C = Cfg<kPair>;
  constexpr int kStages = C::kStages;
  constexpr int kBStage = C::kBStage;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + kStages * kABytes;
  StageExtra* sX = reinterpret_cast<StageExtra*>(sB + kStages * kBStage);
  SmemCtl* ctl = reinterpret_cast<SmemCtl*>((reinterpret_cast<uintptr_t>(sX + kStages) + 127) & ~uintptr_t(127));
  volatile int* abort_flag = &ctl->abort_flag;

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const uint32_t rank = kPair ? cluster_rank() : 0u;       // 0 = leader of the pair
  // work is dealt per CTA, or per pair of CTAs (recomputed where used, to keep registers free)
#define MOE_CTA_ID (kPair ? blockIdx.x / 2u : blockIdx.x)
#define MOE_CTA_COUNT (kPair ? gridDim.x / 2u : gridDim.x)

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&ctl->full[s]), 1);
      mbar_init(smem_u32(&ctl->xfull[s]), 1);
      // MMA commit + every local epilogue warp (block-scaled: the MMA warp
      // alone reads the stage's side data)
      mbar_init(smem_u32(&ctl->empty[s]), kBS ? 1 : 1 + kNumEpiWarps);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&ctl->tfull[b]), 1);
      mbar_init(smem_u32(&ctl->tempty[b]), (kPair ? 2 : 1) * kNumEpiWarps);
    }
    ctl->abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc_k<kPair>(smem_u32(&ctl->tmem_base), kTmemCols);
    tmem_relinquish_k<kPair>();
  }
  pdl_launch_dependents();
  // The plan is an input of the forward, complete before its first launch
  // began, so it is read before the dependency wait; everything the
  // previous kernels of this forward write is read after it.
  int64_t P = *p.num_post_padded;
  if (P < 0) P = 0;
  int64_t nvalid = P / p.block_m;
  if (nvalid > p.nblocks) nvalid = p.nblocks;
  const int64_t ncache = nvalid < kMaxBlocksSmem ? nvalid : kMaxBlocksSmem;
  for (int64_t b = threadIdx.x; b < ncache; b += blockDim.x) ctl->expert[b] = p.expert_ids[b];
  if (kPair) {
    __syncthreads();
    // a block leads a pair when an even number of blocks of its expert
    // precede it; its partner is the next block if it has the same expert
    for (int64_t b = threadIdx.x; b < ncache; b += blockDim.x) {
      const int e = ctl->expert[b];
      int64_t run = 0;
      while (b - run - 1 >= 0 && ctl->expert[b - run - 1] == e) ++run;
      const bool lead = (run & 1) == 0;
      const bool partner = lead && b + 1 < ncache && ctl->expert[b + 1] == e;
      ctl->pairf[b] = static_cast<uint8_t>((lead ? 1 : 0) | (partner ? 2 : 0));
    }
  }
  tc_fence_before();
  __syncthreads();
  if (kPair) cluster_sync();  // the peer's copies and arrivals target initialised barriers
  tc_fence_after();
  const uint32_t tmem_base = ctl->tmem_base;
  const int64_t total = p.nblocks * p.ntiles_n * p.splits;
  // the producer of a single CTA waits after prefetching weights
  if (kPair || warp != 0) pdl_wait();
  // the staging kernel (complete now) stamped this forward's routes with
  // gen + 1; the combine reads the advanced value
  if (kUp && p.gen && blockIdx.x == 0 && threadIdx.x == 64) *p.gen += 1u;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    uint32_t it = 0;
    bool ok = true;
    int64_t tile = MOE_CTA_ID;
    int b = 0, t = 0, sp = 0, e = 0;
    while (tile < total && !tile_coords<kPair>(p, ctl, tile, nvalid, b, t, sp, e)) tile += MOE_CTA_COUNT;
    // Weight tiles of the first ring stages go out before the dependency
    // wait (weights are inputs): their latency overlaps the previous
    // kernel's tail.  Their bytes are added to the stage's transaction count
    // without arriving, so the stage completes only after the arrival below,
    // which also expects the activation rows and side data.
    uint32_t npre = 0;
    if (!kPair) {
      int64_t pt = tile;
      int pb = b, pt_n = t, psp = sp, pe = e;
      int pkb = psp * p.ksplit, pkb1 = min(p.nkb, pkb + p.ksplit);
      while (pt < total && npre < static_cast<uint32_t>(kStages)) {
        if (lane == 0) {
          const uint32_t full = smem_u32(&ctl->full[npre]);
          mbar_expect_tx(full, kBStage);
          int bx = pkb * kTileK, by = pe * p.b_rows + pt_n * kTileN;
          MOE_CHECK_BOX(bx, by, p.nkb * kTileK, static_cast<int64_t>(p.E) * p.b_rows, 16);
          tma_load_2d(smem_u32(sB + npre * kBStage), &tmB, full, bx, by);
        }
        ++npre;
        if (++pkb >= pkb1) {
          pt += MOE_CTA_COUNT;
          while (pt < total && !tile_coords<kPair>(p, ctl, pt, nvalid, pb, pt_n, psp, pe)) pt += MOE_CTA_COUNT;
          pkb = psp * p.ksplit;
          pkb1 = min(p.nkb, pkb + p.ksplit);
        }
      }
      pdl_wait();
    }
    // gather4 path: a tile's plan entries are read one tile ahead
    int ids[4] = {-1, -1, -1, -1};
    if (kUp && !kPair && p.a_gather4 && tile < total) load_ids(p, b, lane, ids);
    const uint32_t lead_full0 = kPair ? mapa_shared(smem_u32(&ctl->full[0]), 0) : smem_u32(&ctl->full[0]);
    while (tile < total && ok) {
      int64_t ntile = tile + MOE_CTA_COUNT;
      int nb = 0, nt = 0, nsp = 0, ne = 0;
      while (ntile < total && !tile_coords<kPair>(p, ctl, ntile, nvalid, nb, nt, nsp, ne)) ntile += MOE_CTA_COUNT;
      // this CTA's plan block; in a pair the second CTA takes the partner block
      const bool partner = kPair && (ctl->pairf[b] & 2);
      const bool has_rows = !kPair || rank == 0 || partner;
      const int mb = b + static_cast<int>(kPair && rank == 1 && partner ? 1 : 0);
      int tok[4] = {0, 0, 0, 0};
      bool mine = false;                 // this lane's four rows hold a route
      uint32_t a_bytes = has_rows ? kABytes : 0u;
      if (kUp && !kPair && p.a_gather4) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const bool route = ids[i] >= 0 && ids[i] < p.R;
          mine |= route;
          tok[i] = route ? ids[i] / p.top_k : 0;
          if (!MOE_IN_BOUNDS(tok[i] < p.a_rows)) tok[i] = 0;
        }
        // only groups with a route are fetched; the other rows keep stale
        // shared memory, whose products land in rows the epilogue ignores
        a_bytes = 512u * static_cast<uint32_t>(__popc(__ballot_sync(0xffffffffu, mine)));
        if (ntile < total) load_ids(p, nb, lane, ids);
      }
      // the leader's barrier counts the operand bytes of both CTAs
      const uint32_t op_bytes = kPair ? (kABytes + (partner ? kABytes : 0u) + 2u * kBStage) : a_bytes + kBStage;
      const uint32_t op_bytes_pre = a_bytes;  // weight tile already expected and in flight
      const int brow = e * p.b_rows + t * kTileN + static_cast<int>(rank) * kBStage / kTileK;
      const int64_t slot0 = static_cast<int64_t>(mb) * p.block_m;
      const int kb0 = sp * p.ksplit;
      const int kb1 = min(p.nkb, kb0 + p.ksplit);
      for (int kb = kb0; kb < kb1; ++kb) {
        const int s = it % kStages;
        const uint32_t ph = (it / kStages) & 1u;
        if (!warp_wait(smem_u32(&ctl->empty[s]), ph ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        const uint32_t full = kPair ? lead_full0 + 8u * s : smem_u32(&ctl->full[s]);
        const uint32_t xfull = smem_u32(&ctl->xfull[s]);
        const bool tile_info = (!kUp || (!kPair && p.splits > 1)) && kb == kb0;
        const uint32_t extra = 512u + 16u + (tile_info ? 1024u : 0u);
        const bool pre = it < npre;
        if (lane == 0) {
          if (!kPair || rank == 0) mbar_arrive_expect_tx(smem_u32(&ctl->full[s]), pre ? op_bytes_pre : op_bytes);
          mbar_arrive_expect_tx(xfull, extra);
        }
        // the small side copies go first: queued behind the operand boxes
        // they would land last and hold up the epilogue, which frees the stage
        if (lane == 0) {
          StageExtra* x = sX + s;
          // (a failing check reads from offset 0 instead, so the stage still completes)
          const bool slots_ok = MOE_IN_BOUNDS(slot0 >= 0 && slot0 % 4 == 0 && slot0 + 128 <= p.cap_pad);
          int64_t as_off = static_cast<int64_t>(kb) * p.cap_pad + slot0;
          if (!slots_ok || !MOE_IN_BOUNDS(kb < p.nkb)) as_off = 0;
          int64_t ws_off = (static_cast<int64_t>(b) * p.ntiles_n + t) * p.nkb + kb;
          if (!MOE_IN_BOUNDS(ws_off < p.nblocks * p.ntiles_n * p.nkb)) ws_off = 0;
          bulk_load(smem_u32(x->a_scale), p.a_scale_t + as_off, 512u, xfull);
          bulk_load(smem_u32(&x->w_scale), p.w_scale_st + ws_off, 16u, xfull);
          if (tile_info) {
            bulk_load(smem_u32(x->tok), p.slot_route + (slots_ok ? slot0 : 0), 512u, xfull);
            bulk_load(smem_u32(x->weight), p.slot_w + (slots_ok ? slot0 : 0), 512u, xfull);
          }
        }
        __syncwarp();
        const uint32_t a_dst = smem_u32(sA + s * kABytes);
        if (kUp && !kPair && p.a_gather4) {
          int gx = kb * kTileK, gy = 0;
          MOE_CHECK_BOX(gx, gy, p.nkb * kTileK, 1, 16);
          if (mine) tma_gather4(a_dst + 512u * lane, &tmA, full, gx, tok[0], tok[1], tok[2], tok[3]);
        } else if (lane == 0 && has_rows) {
          int ax = kb * kTileK, ay = mb * p.block_m;
          MOE_CHECK_BOX(ax, ay, p.nkb * kTileK, p.a_rows, 16);
          if (kPair)
            tma_load_2d_pair(a_dst, &tmA, full, ax, ay);
          else
            tma_load_2d(a_dst, &tmA, full, ax, ay);
        }
        if (lane == 0 && !pre) {
          int bx = kb * kTileK, by = brow;
          MOE_CHECK_BOX(bx, by, p.nkb * kTileK, static_cast<int64_t>(p.E) * p.b_rows, 16);
          if (kPair)
            tma_load_2d_pair(smem_u32(sB + s * kBStage), &tmB, full, bx, by);
          else
            tma_load_2d(smem_u32(sB + s * kBStage), &tmB, full, bx, by);
        }
        ++it;
      }
      tile = ntile;
      b = nb;
      t = nt;
      sp = nsp;
      e = ne;
    }
    if (!ok && lane == 0) {
      // wind down: let the copies already issued land before the CTA exits
      for (uint32_t j = (it > kStages ? it - kStages : 0); j < it; ++j) {
        if (!kPair || rank == 0) drain_wait(smem_u32(&ctl->full[j % kStages]), (j / kStages) & 1u);
        drain_wait(smem_u32(&ctl->xfull[j % kStages]), (j / kStages) & 1u);
      }
    }
  } else if (warp == 1 && kBS) {
    // ------------------------------------------------------------ block-scaled MMA issuer
    // The whole warp turns each slice's FP32 power-of-two scales into UE8M0
    // scale-factor rows in shared memory (lane r: A rows r, 32+r, 64+r, 96+r;
    // B columns 32 i + r, which in the interleaved tile are gate columns for
    // r % 16 < 8 and up columns otherwise); lane 0 copies them into the
    // stage's tensor-memory columns and issues the slice's four MMAs, which
    // accumulate into the tile's one buffer.
    uint8_t* sf_smem = &ctl->u.up.sf[0][0];
    uint32_t it = 0, tcount = 0;
    bool ok = true, bad = false;
    for (int64_t tile = MOE_CTA_ID; tile < total && ok; tile += MOE_CTA_COUNT) {
      int b, t, sp, e;
      if (!tile_coords<kPair>(p, ctl, tile, nvalid, b, t, sp, e)) continue;
      const int kb0 = sp * p.ksplit;
      const int kb1 = min(p.nkb, kb0 + p.ksplit);
      // the accumulator is free once the epilogue has read the previous tile
      if (!warp_wait(smem_u32(&ctl->tempty[0]), (tcount & 1u) ^ 1u, abort_flag)) {
        ok = false;
        break;
      }
      for (int kb = kb0; kb < kb1; ++kb) {
        const int s = it % kStages;
        const uint32_t ph = (it / kStages) & 1u;
        // side data first: the stage (and its scale-factor slot) is free again once it has landed
        if (!warp_wait(smem_u32(&ctl->xfull[s]), ph, abort_flag)) {
          ok = false;
          break;
        }
        const StageExtra* x = sX + s;
        uint8_t* sfa = sf_smem + s * 1024;
        uint8_t* sfb = sfa + 512;
        // (the staging kernel checks the activation scales of the rows that
        // hold a route; pad rows' products are never stored)
        uint32_t wa[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) wa[i] = ue8m0_word(x->a_scale[32 * i + lane]);
        const float4 ws = x->w_scale;
        bad |= !ue8m0_ok(ws.x) || !ue8m0_ok(ws.y);
        const uint32_t wb = ue8m0_word((lane & 8) ? ws.y : ws.x);
        *reinterpret_cast<uint4*>(sfa + 16 * lane) = make_uint4(wa[0], wa[1], wa[2], wa[3]);
        *reinterpret_cast<uint4*>(sfb + 16 * lane) = make_uint4(wb, wb, wb, wb);
        fence_proxy_async_smem();
        __syncwarp();
        int okl = 1;
        if (lane == 0) okl = mbar_wait(smem_u32(&ctl->full[s]), ph, abort_flag) ? 1 : 0;
        if (!__shfl_sync(0xffffffffu, okl, 0)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          tc_fence_after();
          const uint32_t tsf = tmem_base + kSfTmemCol + 16u * s;
          tmem_cp_32x128b_warpx4(tsf, rows16_desc(smem_u32(sfa)));       // A rows 0..127
          tmem_cp_32x128b_warpx4(tsf + 4, rows16_desc(smem_u32(sfb)));   // B columns 0..127
          tmem_cp_32x128b_warpx4(tsf + 8, rows16_desc(smem_u32(sfb)));   // B columns 128..255 (same pattern)
          const uint32_t a0 = smem_u32(sA + s * kABytes);
          const uint32_t b0 = smem_u32(sB + s * kBStage);
#pragma unroll
          for (int kk = 0; kk < kTileK / 32; ++kk)
            umma_mx8(tmem_base, sw128_kmajor_desc(a0 + 32u * kk), sw128_kmajor_desc(b0 + 32u * kk), kIdescMx, tsf,
                     tsf + 4, (kb > kb0 || kk > 0) ? 1u : 0u);
          umma_commit(smem_u32(&ctl->empty[s]));
          if (kb == kb1 - 1) umma_commit(smem_u32(&ctl->tfull[0]));
        }
        __syncwarp();
        ++it;
      }
      ++tcount;
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) report(p.status, MOE_DEV_BAD_SCALE);
    // no MMA or copy may still be writing tensor memory when it is released:
    // the last slice's commit on its stage's empty barrier covers them all
    if (lane == 0 && it > 0) drain_wait(smem_u32(&ctl->empty[(it - 1) % kStages]), ((it - 1) / kStages) & 1u);
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (leader of a pair)
    if (lane == 0 && rank == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int64_t tile = MOE_CTA_ID; tile < total && ok; tile += MOE_CTA_COUNT) {
        int b, t, sp, e;
        if (!tile_coords<kPair>(p, ctl, tile, nvalid, b, t, sp, e)) continue;
        const int kb0 = sp * p.ksplit;
        const int kb1 = min(p.nkb, kb0 + p.ksplit);
        for (int kb = kb0; kb < kb1; ++kb) {
          const int s = it % kStages;
          const uint32_t ph = (it / kStages) & 1u;
          const uint32_t tb = it & 1u;
          const uint32_t tph = (it >> 1) & 1u;
          if (!mbar_wait(smem_u32(&ctl->full[s]), ph, abort_flag) ||
              !mbar_wait(smem_u32(&ctl->tempty[tb]), tph ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(sA + s * kABytes);
          const uint32_t b0 = smem_u32(sB + s * kBStage);
          const uint32_t d = tmem_base + tb * kTileN;
#pragma unroll
          for (int kk = 0; kk < kTileK / 32; ++kk) {
            if (kPair)
              umma_f8_pair(d, sw128_kmajor_desc(a0 + 32u * kk), sw128_kmajor_desc(b0 + 32u * kk), C::kIdesc,
                           kk > 0 ? 1u : 0u);
            else
              umma_f8(d, sw128_kmajor_desc(a0 + 32u * kk), sw128_kmajor_desc(b0 + 32u * kk), C::kIdesc,
                      kk > 0 ? 1u : 0u);
          }
          if (kPair) {
            umma_commit_pair(smem_u32(&ctl->empty[s]));
            umma_commit_pair(smem_u32(&ctl->tfull[tb]));
          } else {
            umma_commit(smem_u32(&ctl->empty[s]));
            umma_commit(smem_u32(&ctl->tfull[tb]));
          }
          ++it;
        }
      }
      // no MMA may still be writing TMEM when it is released
      if (it > 0) drain_wait(smem_u32(&ctl->tfull[(it - 1) & 1u]), ((it - 1) >> 1) & 1u);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;
    const int row = quarter * 32 + lane;
    const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
    uint32_t it = 0;
    int tcount = 0;
    bool ok = true;
    for (int64_t tile = MOE_CTA_ID; tile < total; tile += MOE_CTA_COUNT) {
      int b, t, sp, e;
      if (!tile_coords<kPair>(p, ctl, tile, nvalid, b, t, sp, e)) {
        if (warp == 2 && lane == 0 && rank == 0 && t == 0 && sp == 0 && static_cast<int64_t>(b) < nvalid &&
            (!kPair || (ctl->pairf[b] & 1))) {
          const int bad = block_expert(p, ctl, b);
          if (bad != -1) report(p.status, MOE_DEV_BAD_EXPERT);
        }
        continue;
      }
      int tok = -1;
      float wr = 0.f;

      float acc[128];
#pragma unroll
      for (int c = 0; c < 128; ++c) acc[c] = 0.f;

      const int kb0 = sp * p.ksplit;
      const int kb1 = min(p.nkb, kb0 + p.ksplit);
      if (kBS) {
        // the tile's sum, scaled by the tensor core, in the one accumulator
        if (ok) ok = warp_wait(smem_u32(&ctl->tfull[0]), tcount & 1u, abort_flag);
        if (ok) {
          tc_fence_after();
#pragma unroll
          for (int ch = 0; ch < 8; ++ch) {
            uint32_t v[16];
            tmem_ld_32x32b_x16(lane_base + 128u * half + 16u * ch, v);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) acc[16 * ch + i] = __uint_as_float(v[i]);
          }
          tc_fence_before();
        }
        __syncwarp();
        if (ok && lane == 0) mbar_arrive(smem_u32(&ctl->tempty[0]));
        if (p.splits > 1) {
          const int64_t slot = static_cast<int64_t>(b) * p.block_m + row;
          ctl->row_tok[row] = (row < p.block_m && MOE_IN_BOUNDS(slot < p.cap_pad)) ? p.slot_route[slot] : -1;
        }
      }
      for (int kb = kb0; kb < (kBS ? kb0 : kb1); ++kb) {
        const int s = it % kStages;
        const uint32_t ph = (it / kStages) & 1u;
        const uint32_t tb = it & 1u;
        const uint32_t tph = (it >> 1) & 1u;
        // the slice's scales (and the tile's row data) arrive with the stage
        float s0 = 0.f, s1 = 0.f;
        if (ok) ok = warp_wait(smem_u32(&ctl->xfull[s]), ph, abort_flag);
        if (ok) {
          const StageExtra* x = sX + s;
          const float as = x->a_scale[row];
          const float4 ws = x->w_scale;
          if (kUp) {
            s0 = __fmul_rn(as, ws.x);  // gate block
            s1 = __fmul_rn(as, ws.y);  // up block
          } else {
            s0 = __fmul_rn(as, half == 0 ? ws.x : ws.y);
          }
          if (kb == kb0) {
            if (!kUp) {
              tok = x->tok[row];
              wr = x->weight[row];
            } else if (!kPair && p.splits > 1) {
              ctl->row_tok[row] = x->tok[row];  // read back at the tile end (keeps registers free)
            }
          }
        }
        __syncwarp();
        if (ok && lane == 0) mbar_arrive(smem_u32(&ctl->empty[s]));
        if (ok) ok = warp_wait(smem_u32(&ctl->tfull[tb]), tph, abort_flag);
        if (ok) {
          tc_fence_after();
#pragma unroll
          for (int ch = 0; ch < 8; ++ch) {
            uint32_t v[16];
            tmem_ld_32x32b_x16(lane_base + tb * kTileN + 128u * half + 16u * ch, v);
            tmem_wait_ld();
            // packed FP32 FMAs, two columns each (same rounding as two fmaf)
#pragma unroll
            for (int i = 0; i < 16; i += 2) {
              const float sc = (kUp && (i & 8)) ? s1 : s0;  // up kernel: gate columns 0-7, up columns 8-15
              const float2 r = __ffma2_rn(make_float2(__uint_as_float(v[i]), __uint_as_float(v[i + 1])),
                                          make_float2(sc, sc), make_float2(acc[16 * ch + i], acc[16 * ch + i + 1]));
              acc[16 * ch + i] = r.x;
              acc[16 * ch + i + 1] = r.y;
            }
          }
          tc_fence_before();
        }
        __syncwarp();
        if (ok && lane == 0) {
          if (kPair && rank == 1)
            mbar_arrive_cluster(mapa_shared(smem_u32(&ctl->tempty[tb]), 0));
          else
            mbar_arrive(smem_u32(&ctl->tempty[tb]));
        }
        ++it;
      }

      // this CTA's plan block (in a pair the second CTA takes the partner
      // block), its row validity and plan slot; evaluated where needed
#define MOE_HAS_ROWS (!kPair || rank == 0 || (ctl->pairf[b] & 2))
#define MOE_RVALID (MOE_HAS_ROWS && row < p.block_m)
#define MOE_SLOT (static_cast<int64_t>(b + ((kPair && rank == 1) ? 1 : 0)) * p.block_m + row)
      bool have = true;  // this CTA holds the tile's complete sum
      if (kUp && !kPair && p.splits > 1) {
        // split K: add this split's partial into the tile's zeroed sum; the
        // split that arrives last reads the total back and finishes the tile.
        // Every split takes its ticket, even one whose waits ran out (it adds
        // nothing then), and the last one clears all the tile's rows, so the
        // tickets and sums are back to zero after any forward.
        const int64_t sum_row = (static_cast<int64_t>(b) * p.ntiles_n + t) * p.block_m + (MOE_RVALID ? row : 0);
        const bool sum_ok = MOE_IN_BOUNDS(sum_row < p.nblocks * p.ntiles_n * p.block_m);
        const bool live = ok && sum_ok && MOE_RVALID && ctl->row_tok[row] >= 0;
        float* srow = p.usum + (sum_ok ? sum_row : 0) * kTileN + 128 * half;
        if (live) {
#pragma unroll
          for (int c = 0; c < 128; c += 4) red_add_v4(srow + c, acc[c], acc[c + 1], acc[c + 2], acc[c + 3]);
        }
        __threadfence();
        named_barrier(1, 32 * kNumEpiWarps);
        if (warp == 2 && lane == 0) {
          int64_t cnt_off = static_cast<int64_t>(b) * p.ntiles_n + t;
          if (!MOE_IN_BOUNDS(cnt_off < p.nblocks * p.ntiles_n)) cnt_off = 0;
          int32_t* cnt = p.ucnt + cnt_off;
          const int old = atomicAdd(cnt, 1);
          const bool last = old == p.splits - 1;
          if (last) *cnt = 0;
          ctl->last_flag = last ? 1 : 0;
        }
        named_barrier(1, 32 * kNumEpiWarps);
        have = ctl->last_flag != 0;
        if (have) {
          __threadfence();
          if (MOE_RVALID && sum_ok) {
#pragma unroll
            for (int c = 0; c < 128; c += 4) {
              const float4 v = __ldcg(reinterpret_cast<const float4*>(srow + c));
              acc[c] = v.x;
              acc[c + 1] = v.y;
              acc[c + 2] = v.z;
              acc[c + 3] = v.w;
              *reinterpret_cast<float4*>(srow + c) = make_float4(0.f, 0.f, 0.f, 0.f);
            }
          }
        }
      }
      if (kUp && have) {
        // SwiGLU on the 64 (gate, up) pairs this thread holds, then the
        // per-token 1x128 requant shared with the partner warp (other half).
        float amax = 0.f;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float h = __fmul_rn(silu_f32(acc[16 * q + j]), acc[16 * q + 8 + j]);
            acc[8 * q + j] = h;  // compact in place: slot 8q+j is free once read
            amax = fmaxf(amax, fabsf(h));
          }
        }
        ctl->u.up.xchg[tcount & 1][half][row] = amax;
        named_barrier(1, 32 * kNumEpiWarps);
        amax = fmaxf(amax, ctl->u.up.xchg[tcount & 1][half ^ 1][row]);
        const float s = __fdiv_rn(amax, 448.0f);
        // h / s as h * (1/s): the two roundings can move a value across an
        // E4M3 rounding midpoint only when it lies within an ulp of it
        const float inv = s > 0.f ? __frcp_rn(s) : 0.f;
        uint32_t packed[16];
#pragma unroll
        for (int w = 0; w < 16; ++w) {
          const uint16_t lo = cvt_e4m3x2(__fmul_rn(acc[4 * w + 0], inv), __fmul_rn(acc[4 * w + 1], inv));
          const uint16_t hi = cvt_e4m3x2(__fmul_rn(acc[4 * w + 2], inv), __fmul_rn(acc[4 * w + 3], inv));
          packed[w] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
        }
        // The codes leave through tensor stores of whole row boxes: the warp's
        // 32 rows are consecutive plan slots; boxes stop at the plan block's
        // last row (the next block's slots belong to another CTA).
        {
          const int64_t wslot = MOE_SLOT - lane;  // the warp's first row
          int nvr = MOE_HAS_ROWS ? p.block_m - 32 * (warp & 3) : 0;
          nvr = nvr < 0 ? 0 : (nvr > 32 ? 32 : nvr);
          if (!ok) nvr = 0;
          uint8_t* stage = ctl->u.up.qst[warp - 2];
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            if (nvr > 0) {
              if (r > 0) {
                if (lane == 0) bulk_wait_read_all();
                __syncwarp();
              }
              *reinterpret_cast<uint4*>(stage + 32 * lane) =
                  make_uint4(packed[8 * r], packed[8 * r + 1], packed[8 * r + 2], packed[8 * r + 3]);
              *reinterpret_cast<uint4*>(stage + 32 * lane + 16) =
                  make_uint4(packed[8 * r + 4], packed[8 * r + 5], packed[8 * r + 6], packed[8 * r + 7]);
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                for (int r0 = 0; r0 < nvr; r0 += p.qbox) {
                  int qx = 128 * t + 64 * half + 32 * r, qy = static_cast<int>(wslot) + r0;
                  MOE_CHECK_BOX(qx, qy, p.I, p.q_rows - p.qbox + 1, 16);
                  tma_store_2d(&tmQ, smem_u32(stage + 32 * r0), qx, qy);
                }
                bulk_commit();
              }
            }
          }
          if (nvr > 0 && lane == 0) bulk_wait_read_all();  // the stage is rewritten by the next tile
          __syncwarp();
        }
        if (ok && MOE_RVALID && MOE_IN_BOUNDS(MOE_SLOT < p.q_rows && MOE_SLOT < p.cap_pad)) {
          const int64_t slot = MOE_SLOT;
          const int64_t qoff = slot * p.I + 128 * t + 64 * half;
          if (half == 0) p.s_inter_t[static_cast<int64_t>(t) * p.cap_pad + slot] = s;
          if (p.dbg_q) {
            uint4* ddst = reinterpret_cast<uint4*>(p.dbg_q + qoff);
#pragma unroll
            for (int w = 0; w < 4; ++w)
              ddst[w] = make_uint4(packed[4 * w], packed[4 * w + 1], packed[4 * w + 2], packed[4 * w + 3]);
            if (half == 0) p.dbg_s[slot * (p.I / 128) + t] = s;
          }
        }
      } else if (!kUp) {
        // this row's contribution y * w for its route (`tok` holds the route
        // id), rounded to BF16: 128 columns = 256 contiguous bytes
        // Stored transposed through shared memory, 32 columns at a time, so
        // one instruction writes 8 rows x 64 contiguous bytes.
        const int hblk = 2 * t + half;
        const bool live = ok && hblk < p.H / 128 && MOE_RVALID && tok >= 0;
        if (__any_sync(0xffffffffu, live)) {
          uint32_t(*buf)[20] = ctl->u.yt[warp - 2];
          const int sub = lane >> 2, c16 = lane & 3;  // row 8 i + sub, 16-byte segment c16 of 64
          int rts[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) rts[i] = __shfl_sync(0xffffffffu, live ? tok : -1, 8 * i + sub);
#pragma unroll
          for (int ch = 0; ch < 4; ++ch) {
#pragma unroll
            for (int w = 0; w < 16; ++w) {
              const int c = 32 * ch + 2 * w;
              const __nv_bfloat162 v = __floats2bfloat162_rn(__fmul_rn(acc[c], wr), __fmul_rn(acc[c + 1], wr));
              buf[lane][w] = *reinterpret_cast<const uint32_t*>(&v);
            }
            __syncwarp();
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              if (rts[i] >= 0) {
                const uint32_t* src = &buf[8 * i + sub][4 * c16];
                uint4* dst = reinterpret_cast<uint4*>(p.y_out + static_cast<int64_t>(rts[i]) * p.H + hblk * 128 +
                                                      32 * ch + 8 * c16);
                if (MOE_IN_BOUNDS(rts[i] < p.R && hblk * 128 + 32 * ch + 8 * c16 + 8 <= p.H))
                  *dst = make_uint4(src[0], src[1], src[2], src[3]);
              }
            }
            __syncwarp();
          }
        }
      }
      ++tcount;
    }
    // the codes' tensor stores are complete before the grid is (the down
    // kernel reads them after its dependency wait)
    if (kUp && lane == 0) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  if (kPair) cluster_sync();  // neither CTA leaves while the pair still touches its memory
  tc_fence_after();
  if (threadIdx.x == 0 && ctl->abort_flag) report(p.status, MOE_DEV_TIMEOUT);
  if (warp == 1) tmem_dealloc_k<kPair>(tmem_base, kTmemCols);
#undef MOE_CTA_ID
#undef MOE_CTA_COUNT
#undef MOE_HAS_ROWS
#undef MOE_RVALID
#undef MOE_SLOT
}

// Staging for the GEMM kernels (launch 0).  Part 1, one warp per plan slot
// below P: token and route weight of the slot (-1 / 0 for pads), the
// activation scales transposed to [nkb, cap_pad], and for well-filled plans
// the activation row copied into plan order.  Part 2, per plan block below P
// with a valid expert: the 16-byte weight-scale records of every (n tile,
// K slice) of both GEMMs.
struct StageParams {
  const uint8_t* a;
  const float* a_scale;
  const float* topk_w;
  const int32_t* sorted_ids;
  const int32_t* expert_ids;
  const int32_t* num_post_padded;
  const float* w13_scale;
  const float* w2_scale;
  uint8_t* a_sorted;          // nullable: no row copy
  float* as_t;                // [nkb, cap_pad]
  int32_t* slot_route;        // [cap_pad]
  uint32_t* rvalid;           // [R] set to this forward's stamp for each route the plan holds
  const uint32_t* gen;        // stamp of the previous forward (this one's is gen + 1)
  float* slot_w;              // [cap_pad]
  int32_t* status;            // nullable
  int64_t a_rows;             // rows of a_sorted (sorted_cap)
  int check_pow2;             // block-scaled mode: activation scales must be +0 or normal powers of two
  float4* wsu;                // [nblocks, I/128, H/128]
  float4* wsd;                // [nblocks, ceil(H/256), I/128]
  int64_t nblocks;
  int64_t cap_pad;
  int R, top_k, block_m, E, H, I;
  float routed_scale;
};

__global__ void __launch_bounds__(256) stage_kernel(const StageParams p) {
  // Trigger only after the wait: the GEMMs read the plan before their own
  // dependency wait, which is sound once this grid has waited for the
  // (programmatically launched) plan kernels.
  pdl_wait();
  pdl_launch_dependents();
  int64_t P = *p.num_post_padded;
  if (P < 0) P = 0;
  int64_t nvalid = P / p.block_m;
  if (nvalid > p.nblocks) nvalid = p.nblocks;
  const int64_t nslots = nvalid * p.block_m;
  const int lane = threadIdx.x % 32;
  const int64_t gtid = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * (blockDim.x / 32);
  const int nkb = p.H / 128, nib = p.I / 128;
  const int chunks = p.H / 16;
  for (int64_t slot = gtid / 32; slot < nslots; slot += nwarps) {
    if (!MOE_IN_BOUNDS(slot < p.cap_pad)) break;
    const int id = p.sorted_ids[slot];
    const bool route = id >= 0 && id < p.R;
    const int64_t tok = route ? id / p.top_k : 0;
    if (lane == 0) {
      p.slot_route[slot] = route ? id : -1;
      p.slot_w[slot] = route ? __fmul_rn(__ldg(p.topk_w + id), p.routed_scale) : 0.f;
      if (route) p.rvalid[id] = *p.gen + 1u;
    }
    if (!route) continue;
    if (p.a_sorted && MOE_IN_BOUNDS(slot < p.a_rows)) {
      // up to 4 KB of the row in flight per warp (8 loads per lane) before the stores
      const uint4* src = reinterpret_cast<const uint4*>(p.a + tok * p.H);
      uint4* dst = reinterpret_cast<uint4*>(p.a_sorted + slot * p.H);
      for (int c0 = 0; c0 < chunks; c0 += 256) {
        uint4 v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int c = c0 + 32 * j + lane;
          if (c < chunks) v[j] = __ldg(src + c);
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int c = c0 + 32 * j + lane;
          if (c < chunks) dst[c] = v[j];
        }
      }
    }
  }
  // activation scales transposed to [K slice][slot]: a warp per 32
  // consecutive slots, lane = slot, so each slice's 32 scales are one
  // 128-byte store (each lane walks its own token's scale row)
  for (int64_t s0 = gtid / 32 * 32; s0 < nslots; s0 += nwarps * 32) {
    const int64_t slot = s0 + lane;
    int id = -1;
    if (slot < nslots) id = p.sorted_ids[slot];
    const bool route = id >= 0 && id < p.R;
    const float* row = p.a_scale + (route ? static_cast<int64_t>(id / p.top_k) * nkb : 0);
    if (slot < nslots && MOE_IN_BOUNDS(slot < p.cap_pad)) {
      for (int k = 0; k < nkb; ++k) {
        const float v = route ? __ldg(row + k) : 0.f;
        p.as_t[k * p.cap_pad + slot] = v;
        if (route && p.check_pow2 && !ue8m0_ok(v)) report(p.status, MOE_DEV_BAD_SCALE);
      }
    }
  }
  // weight-scale records: a CTA per plan block, its threads over the block's
  // records (no 64-bit divisions)
  const int up_items = nib * nkb;          // (n tile: I/128 of them) x (K slice)
  const int nh = (p.H + 255) / 256;
  const int dn_items = nh * nib;
  const int per_block = up_items + dn_items;
  const int nrb13 = 2 * p.I / 128, nrb2 = p.H / 128;
  for (int64_t b = blockIdx.x; b < nvalid; b += gridDim.x) {
    if (!MOE_IN_BOUNDS(b < p.nblocks)) break;
    const int e = p.expert_ids[b];
    if (e < 0 || e >= p.E) continue;
    for (int j = threadIdx.x; j < per_block; j += blockDim.x) {
      if (j < up_items) {
        const int t = j / nkb, kb = j % nkb;
        const float* base = p.w13_scale + static_cast<int64_t>(e) * nrb13 * nkb;
        p.wsu[b * up_items + j] = make_float4(base[t * nkb + kb], base[(nib + t) * nkb + kb], 0.f, 0.f);
      } else {
        const int jj = j - up_items;
        const int h = jj / nib, ib = jj % nib;
        const float* base = p.w2_scale + static_cast<int64_t>(e) * nrb2 * nib;
        const float lo = base[(2 * h) * nib + ib];
        const float hi = (2 * h + 1 < nrb2) ? base[(2 * h + 1) * nib + ib] : 0.f;
        p.wsd[b * dn_items + jj] = make_float4(lo, hi, 0.f, 0.f);
      }
    }
  }
}

// Combine: out[t] = bf16_rn(f32(out[t]) + sum_j f32(y[t * top_k + j])) over
// the token's routes that the plan holds (their flag carries this forward's
// stamp), in route order.  A warp per (token, 256-column segment); a token's
// routes are adjacent rows of y.  Rows are loaded eight routes at a time
// whether or not the plan holds them (every row lies inside y), so the
// first loads go out together with the flags; rows of routes not held are
// never added.
__device__ __forceinline__ void add_bf16x8(float (&f)[8], const uint4 v) {
  const uint32_t vw[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    f[2 * k] = __fadd_rn(f[2 * k], __uint_as_float(vw[k] << 16));
    f[2 * k + 1] = __fadd_rn(f[2 * k + 1], __uint_as_float(vw[k] & 0xFFFF0000u));
  }
}

__global__ void __launch_bounds__(256) combine_kernel(uint16_t* __restrict__ out, const uint16_t* __restrict__ y,
                                                      const uint32_t* __restrict__ rvalid, const uint32_t* gen,
                                                      int64_t M, int H, int top_k) {
  constexpr int kBatch = 8;
  pdl_launch_dependents();
  pdl_wait();
  const uint32_t stamp = *gen;  // this forward's stamp on the routes its plan holds
  const int lane = threadIdx.x % 32;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * (blockDim.x / 32);
  const int chunks = H / 8;             // 16-byte groups of eight BF16
  const int segs = (chunks + 31) / 32;  // 256-column segments: a warp each
  for (int64_t wi = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) / 32; wi < M * segs; wi += nwarps) {
    const int64_t t = wi / segs;
    const int seg = static_cast<int>(wi - t * segs);
    const int c = 32 * seg + lane;
    const bool in = c < chunks;
    uint4* o4 = reinterpret_cast<uint4*>(out + t * H);
    const uint4* y4 = reinterpret_cast<const uint4*>(y + t * top_k * static_cast<int64_t>(H)) + c;
    const uint32_t* rv = rvalid + t * top_k;
    // flags (top_k <= 64), the out chunk and the first batch of rows
    const uint32_t fl0 = lane < top_k ? rv[lane] : 0u;
    const uint32_t fl1 = lane + 32 < top_k ? rv[lane + 32] : 0u;
    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
    const uint4 o = in ? o4[c] : zero;
    uint4 v[kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) v[j] = (in && j < top_k) ? __ldcs(y4 + static_cast<int64_t>(j) * chunks) : zero;
    const unsigned vm0 = __ballot_sync(0xffffffffu, lane < top_k && fl0 == stamp);
    const unsigned vm1 = __ballot_sync(0xffffffffu, lane + 32 < top_k && fl1 == stamp);
    const unsigned long long vm = (static_cast<unsigned long long>(vm1) << 32) | vm0;
    float f[8];
    const uint32_t ow[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      f[2 * k] = __uint_as_float(ow[k] << 16);
      f[2 * k + 1] = __uint_as_float(ow[k] & 0xFFFF0000u);
    }
    for (int j0 = 0; j0 < top_k; j0 += kBatch) {
      if (j0 > 0) {
#pragma unroll
        for (int j = 0; j < kBatch; ++j)
          v[j] = (in && j0 + j < top_k) ? __ldcs(y4 + static_cast<int64_t>(j0 + j) * chunks) : zero;
      }
#pragma unroll
      for (int j = 0; j < kBatch; ++j)
        if ((vm >> (j0 + j)) & 1ull) add_bf16x8(f, v[j]);
    }
    if (in) {
      uint32_t r[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const __nv_bfloat162 b = __floats2bfloat162_rn(f[2 * k], f[2 * k + 1]);
        r[k] = *reinterpret_cast<const uint32_t*>(&b);
      }
      o4[c] = make_uint4(r[0], r[1], r[2], r[3]);
    }
  }
}


// Self-test of the failure detection.  Warp 0 waits, through the pipelines'
// bounded wait, on an mbarrier that nothing arrives at, giving up after
// `limit_ns`; warp 1 waits on a second such barrier with the pipelines'
// normal limit and must stop as soon as warp 0 raises the CTA's abort flag.
// The CTA then reports MOE_DEV_TIMEOUT as a GEMM CTA whose wait ran out does.
// elapsed_ns[w] receives how long warp w waited.
__global__ void __launch_bounds__(64, 1)
    wait_selftest_kernel(int32_t* status, unsigned long long limit_ns, unsigned long long* elapsed_ns) {
  __shared__ __align__(8) uint64_t bars[2];
  __shared__ int abort_flag;
  const int warp = threadIdx.x / 32;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bars[0]), 1);
    mbar_init(smem_u32(&bars[1]), 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  const unsigned long long t0 = global_timer_ns();
  const bool ok = warp == 0 ? warp_wait(smem_u32(&bars[0]), 0, &abort_flag, limit_ns)
                            : warp_wait(smem_u32(&bars[1]), 0, &abort_flag);
  const unsigned long long t1 = global_timer_ns();
  if ((threadIdx.x & 31) == 0) elapsed_ns[warp] = ok ? 0ull : t1 - t0;
  __syncthreads();
  if (threadIdx.x == 0 && abort_flag) report(status, MOE_DEV_TIMEOUT);
}

// Activation rows are copied into plan order when plan blocks are well
// filled (at least 8 routes per touched expert on average): tile::gather4
// moves one 128-byte row per ~35 cycles per SM on GB300, far below the rate
// of 2D boxes, and would fetch every row once per 256-wide N tile.  Sparse
// (decode-sized) plans keep gather4 and fetch only groups holding a route.
bool use_pregather(int64_t R, int E) {
  const int64_t nonempty = R < E ? R : E;
  return nonempty > 0 && R >= 8 * nonempty;
}

// Plan blocks that can hold work: P <= R + min(E, R) * (block_m - 1).
int64_t block_bound(int64_t R, int E, int block_m) {
  const int64_t nonempty = R < E ? R : E;
  return ceil_div(R + nonempty * (block_m - 1), block_m);
}

// Split K is available when the gate/up GEMM has fewer tiles than a GB300
// has SMs (decode-sized plans); the workspace then holds the partial sums.
constexpr int64_t kSplitTileLimit = 256;

// The automatic choice takes the vector path up to this many routes (at
// 72 routes the tensor-core tiles are still faster).
constexpr int64_t kVecAutoRoutes = 32;

struct WsLayout {
  size_t y_off, rv_off, gen_off, h_off, q_off, st_off, ast_off, tok_off, w_off, wsu_off, wsd_off, a_off, usum_off, ucnt_off, total;
  int64_t cap_pad, nblocks;
  bool pregather, splitk;
};

WsLayout ws_layout(int64_t M, int H, int I, int E, int top_k, int block_m, int64_t sorted_cap) {
  WsLayout l;
  const int64_t R = M * top_k;
  l.pregather = use_pregather(R, E);
  l.cap_pad = round_up(sorted_cap + kRowPad, 8);  // keeps every 512-byte slice 16-byte aligned
  l.nblocks = block_bound(R, E, block_m);
  if (l.nblocks > sorted_cap / block_m) l.nblocks = sorted_cap / block_m;
  const int nkb = H / 128, nib = I / 128, nh = (H + 255) / 256;
  size_t off = 0;
  auto take = [&](int64_t bytes) {
    const size_t at = off;
    off += static_cast<size_t>(round_up(bytes, 256));
    return at;
  };
  l.y_off = take(R * H * 2);  // BF16 route contributions, by route id
  l.rv_off = take(R * 4);     // route flags: the stamp of the last forward whose plan held the route
  l.gen_off = take(4);        // the last forward's stamp
  // vector path: silu(gate) * up in FP32 by route id
  l.h_off = take(vector_path_supported(M, R, H, I) ? R * I * 4 : 0);
  l.q_off = take(sorted_cap * I);
  l.st_off = take(static_cast<int64_t>(nib) * l.cap_pad * 4);
  l.ast_off = take(static_cast<int64_t>(nkb) * l.cap_pad * 4);
  l.tok_off = take(l.cap_pad * 4);
  l.w_off = take(l.cap_pad * 4);
  l.wsu_off = take(l.nblocks * nib * nkb * 16);
  l.wsd_off = take(l.nblocks * nh * nib * 16);
  l.a_off = take(l.pregather ? sorted_cap * H : 0);
  l.splitk = l.nblocks * nib < kSplitTileLimit;
  l.usum_off = take(l.splitk ? l.nblocks * nib * block_m * 256 * 4 : 0);
  l.ucnt_off = take(l.splitk ? l.nblocks * nib * 4 : 0);
  l.total = off;
  return l;
}


// Clusters of two CTAs that the GPU holds at once.  GPCs need not have an
// even number of SMs, so this can be below SMs / 2; a persistent grid larger
// than it would run its last clusters as a second wave.
int max_pair_clusters(int device, int sms) {
  static std::mutex mu;
  static int cached[64] = {};
  std::lock_guard<std::mutex> lock(mu);
  if (cached[device] > 0) return cached[device];
  int best = sms / 2;
  for (int up = 0; up < 2; ++up) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (sms / 2));
    cfg.blockDim = dim3(kNumThreads);
    cfg.dynamicSmemBytes = smem_bytes<true>();
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    const cudaError_t err =
        up ? cudaOccupancyMaxActiveClusters(&n, moe_gemm_kernel<true, true>, &cfg)
           : cudaOccupancyMaxActiveClusters(&n, moe_gemm_kernel<false, true>, &cfg);
    if (err != cudaSuccess || n <= 0) {
      cudaGetLastError();
      return 0;
    }
    if (n < best) best = n;
  }
  cached[device] = best;
  return best;
}

bool set_smem_attrs(int device) {
  static std::mutex mu;
  static bool done[64] = {};
  std::lock_guard<std::mutex> lock(mu);
  if (done[device]) return true;
  if (cudaFuncSetAttribute(moe_gemm_kernel<true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem_bytes<false>())) != cudaSuccess ||
      cudaFuncSetAttribute(moe_gemm_kernel<false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem_bytes<false>())) != cudaSuccess ||
      cudaFuncSetAttribute(moe_gemm_kernel<true, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem_bytes<true>())) != cudaSuccess ||
      cudaFuncSetAttribute(moe_gemm_kernel<false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem_bytes<true>())) != cudaSuccess ||
      cudaFuncSetAttribute(moe_gemm_kernel<true, false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem_bytes<false>())) != cudaSuccess)
    return false;
  done[device] = true;
  return true;
}

}  // namespace
}  // namespace moe

extern "C" {

size_t moe_forward_workspace_size(int64_t M, int H, int I, int E, int top_k, int block_m, int64_t sorted_cap) {
  if (M < 0 || H < 0 || I < 0 || E < 1 || top_k < 1 || block_m < 1 || sorted_cap < 0) return 0;
  return moe::ws_layout(M, H, I, E, top_k, block_m, sorted_cap).total;
}

moe_status moe_selftest_wait_timeout(uint32_t limit_us, int32_t* device_status, uint64_t* elapsed_ns,
                                     moe_stream_t stream) {
  using namespace moe;
  if (!device_status || !elapsed_ns) return MOE_ERR_NULL;
  if (limit_us < 1 || limit_us > 1000000) return MOE_ERR_SHAPE;
  DeviceInfo dev;
  if (current_device(&dev) != MOE_OK) return MOE_ERR_CUDA;
  if (!on_device(device_status, dev.device) || !on_device(elapsed_ns, dev.device)) return MOE_ERR_DEVICE;
  wait_selftest_kernel<<<1, 64, 0, stream>>>(device_status, 1000ull * limit_us,
                                             reinterpret_cast<unsigned long long*>(elapsed_ns));
  MOE_CUDA_TRY(cudaGetLastError());
  MOE_CUDA_TRY(cudaStreamSynchronize(stream));
  int32_t st = 0;
  MOE_CUDA_TRY(cudaMemcpy(&st, device_status, sizeof(st), cudaMemcpyDeviceToHost));
  return (st & MOE_DEV_TIMEOUT) ? MOE_ERR_TIMEOUT : MOE_OK;
}

moe_status moe_fp8_block_scale_forward(const moe_fwd_args* a, moe_stream_t stream) {
  using namespace moe;
  if (!a) return MOE_ERR_NULL;
  if (a->M < 0 || a->H < 128 || a->H % 128 || a->I < 128 || a->I % 128 || a->E < 1 || a->top_k < 1 ||
      a->top_k > 64)
    return MOE_ERR_SHAPE;
  if (a->block_m < 8 || a->block_m > 128 || a->block_m % 8) return MOE_ERR_SHAPE;
  if (a->tile_mode != MOE_TILE_AUTO && a->tile_mode != MOE_TILE_SINGLE && a->tile_mode != MOE_TILE_PAIR &&
      a->tile_mode != MOE_TILE_VECTOR)
    return MOE_ERR_SHAPE;
  if (a->scale_mode != MOE_SCALES_FP32 && a->scale_mode != MOE_SCALES_UE8M0) return MOE_ERR_SHAPE;
  if (a->blocks_cap < 1 || a->sorted_cap < a->blocks_cap * a->block_m) return MOE_ERR_CAPACITY;
  const int64_t R = a->M * a->top_k;
  if (R >= (int64_t(1) << 31) - 1 || static_cast<int64_t>(a->E) * 2 * a->I >= (int64_t(1) << 31) ||
      static_cast<int64_t>(a->E) * a->H >= (int64_t(1) << 31) || a->sorted_cap >= (int64_t(1) << 30))
    return MOE_ERR_SHAPE;
  const bool vec_ok = vector_path_supported(a->M, R, a->H, a->I);
  if (a->tile_mode == MOE_TILE_VECTOR && !vec_ok) return MOE_ERR_SHAPE;
  if (a->M == 0) return MOE_OK;
  if (!a->a || !a->a_scale || !a->w13 || !a->w13_scale || !a->w2 || !a->w2_scale || !a->topk_weights ||
      !a->sorted_token_ids || !a->expert_ids || !a->num_tokens_post_padded || !a->out || !a->workspace)
    return MOE_ERR_NULL;
  if ((a->debug_q_inter == nullptr) != (a->debug_s_inter == nullptr)) return MOE_ERR_NULL;
  if (!aligned16(a->a) || !aligned16(a->w13) || !aligned16(a->w2) || !aligned16(a->workspace) ||
      !aligned16(a->out) || (a->debug_q_inter && !aligned16(a->debug_q_inter)))
    return MOE_ERR_ALIGN;
  const WsLayout wl = ws_layout(a->M, a->H, a->I, a->E, a->top_k, a->block_m, a->sorted_cap);
  if (a->workspace_bytes < wl.total) return MOE_ERR_CAPACITY;

  DeviceInfo dev;
  if (current_device(&dev) != MOE_OK) return MOE_ERR_CUDA;
  if (dev.major != 10 || dev.minor != 3) return MOE_ERR_DEVICE;
  const void* ptrs[] = {a->a, a->a_scale, a->w13, a->w13_scale, a->w2, a->w2_scale, a->topk_weights,
                        a->sorted_token_ids, a->expert_ids, a->num_tokens_post_padded, a->out, a->workspace};
  for (const void* ptr : ptrs)
    if (!on_device(ptr, dev.device)) return MOE_ERR_DEVICE;
  if (a->device_status && !on_device(a->device_status, dev.device)) return MOE_ERR_DEVICE;
  if (a->debug_q_inter && (!on_device(a->debug_q_inter, dev.device) || !on_device(a->debug_s_inter, dev.device)))
    return MOE_ERR_DEVICE;
  if (!set_smem_attrs(dev.device)) return MOE_ERR_CUDA;

  uint8_t* ws = static_cast<uint8_t*>(a->workspace);
  uint16_t* yr = reinterpret_cast<uint16_t*>(ws + wl.y_off);
  uint32_t* rvalid = reinterpret_cast<uint32_t*>(ws + wl.rv_off);
  uint32_t* gen = reinterpret_cast<uint32_t*>(ws + wl.gen_off);
  uint8_t* q_inter = ws + wl.q_off;
  float* s_inter_t = reinterpret_cast<float*>(ws + wl.st_off);
  float* as_t = reinterpret_cast<float*>(ws + wl.ast_off);
  int32_t* slot_route = reinterpret_cast<int32_t*>(ws + wl.tok_off);
  float* slot_w = reinterpret_cast<float*>(ws + wl.w_off);
  float4* wsu = reinterpret_cast<float4*>(ws + wl.wsu_off);
  float4* wsd = reinterpret_cast<float4*>(ws + wl.wsd_off);
  uint8_t* a_sorted = wl.pregather ? ws + wl.a_off : nullptr;

  const int N = 2 * a->I;
  int64_t nblocks = wl.nblocks;
  if (nblocks > a->blocks_cap) nblocks = a->blocks_cap;
  cudaEvent_t const* ev = reinterpret_cast<cudaEvent_t const*>(a->profile_events);

  // Sparse plans (a few routes per touched expert) take the vector path.
  const bool use_vec = vec_ok && (a->tile_mode == MOE_TILE_VECTOR ||
                                  (a->tile_mode == MOE_TILE_AUTO && R <= kVecAutoRoutes));
  if (use_vec) {
    float* hbuf = reinterpret_cast<float*>(ws + wl.h_off);
    VecUpParams vu{};
    vu.a = a->a;
    vu.a_scale = a->a_scale;
    vu.w13 = a->w13;
    vu.w13_scale = a->w13_scale;
    vu.w2 = a->w2;
    vu.sorted_ids = a->sorted_token_ids;
    vu.expert_ids = a->expert_ids;
    vu.num_post_padded = a->num_tokens_post_padded;
    vu.h = hbuf;
    vu.status = a->device_status;
    vu.nblocks = nblocks;
    vu.R = static_cast<int>(R);
    vu.top_k = a->top_k;
    vu.block_m = a->block_m;
    vu.E = a->E;
    vu.H = a->H;
    vu.I = a->I;
    VecDownParams vd{};
    vd.h = hbuf;
    vd.w2 = a->w2;
    vd.w2_scale = a->w2_scale;
    vd.topk_w = a->topk_weights;
    vd.sorted_ids = a->sorted_token_ids;
    vd.expert_ids = a->expert_ids;
    vd.num_post_padded = a->num_tokens_post_padded;
    vd.out = a->out;
    vd.dbg_q = a->debug_q_inter;
    vd.dbg_s = a->debug_s_inter;
    vd.nblocks = nblocks;
    vd.R = static_cast<int>(R);
    vd.top_k = a->top_k;
    vd.block_m = a->block_m;
    vd.E = a->E;
    vd.H = a->H;
    vd.I = a->I;
    vd.routed_scale = a->routed_scale;
    if (ev) MOE_CUDA_TRY(cudaEventRecord(ev[0], stream));
    const moe_status st = launch_vector_path(vu, vd, stream, ev);
    if (st != MOE_OK) return st;
    if (ev) MOE_CUDA_TRY(cudaEventRecord(ev[4], stream));
    return MOE_OK;
  }
  // CTA pairs (cta_group::2) need the activation rows in plan order and the
  // expert and pair tables in shared memory.  Each SM then streams half of
  // every weight tile, but per K slice the pair runs no faster than a single
  // CTA: the slice's FP32 promotion in the epilogue, not the operand stream,
  // paces the two TMEM buffers.  So the automatic choice stays single.
  // Power-of-two scales on both operands: the gate/up GEMM applies them in
  // the tensor core (single CTAs; a pair request runs single CTAs then).
  const bool block_scaled = a->scale_mode == MOE_SCALES_UE8M0;
  const bool want_pair = a->tile_mode == MOE_TILE_PAIR && !block_scaled;
  const int pair_clusters =
      want_pair && wl.pregather && nblocks <= kMaxBlocksSmem ? max_pair_clusters(dev.device, dev.sms) : 0;
  const bool pair = pair_clusters > 0;
  const uint32_t wbox = pair ? kTileN / 2 : kTileN;
  CUtensorMap tm_a, tm_w13, tm_q, tm_w2;
  const CUresult ra = wl.pregather
                          ? encode_tensor_map_2d(&tm_a, a_sorted, a->H, a->sorted_cap, a->H, 128, 128,
                                                 CU_TENSOR_MAP_SWIZZLE_128B)
                          : encode_tensor_map_2d(&tm_a, a->a, a->H, a->M, a->H, 128, 1, CU_TENSOR_MAP_SWIZZLE_128B);
  if (ra != CUDA_SUCCESS ||
      encode_tensor_map_2d(&tm_w13, a->w13, a->H, static_cast<uint64_t>(a->E) * N, a->H, 128, wbox,
                           CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS ||
      encode_tensor_map_2d(&tm_q, q_inter, a->I, a->sorted_cap, a->I, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B) !=
          CUDA_SUCCESS ||
      encode_tensor_map_2d(&tm_w2, a->w2, a->I, static_cast<uint64_t>(a->E) * a->H, a->I, 128, wbox,
                           CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
    return MOE_ERR_CUDA;
  // tensor stores of the intermediate codes: boxes of 32 codes x qbox rows,
  // qbox the largest of 32, 16, 8 that divides block_m
  const int qbox = a->block_m % 32 == 0 ? 32 : (a->block_m % 16 == 0 ? 16 : 8);
  CUtensorMap tm_qs;
  if (encode_tensor_map_2d(&tm_qs, q_inter, a->I, a->sorted_cap, a->I, 32, static_cast<uint32_t>(qbox),
                           CU_TENSOR_MAP_SWIZZLE_NONE) != CUDA_SUCCESS)
    return MOE_ERR_CUDA;

  if (ev) MOE_CUDA_TRY(cudaEventRecord(ev[0], stream));
  if (nblocks > 0) {
    StageParams sp{};
    sp.a = a->a;
    sp.a_scale = a->a_scale;
    sp.topk_w = a->topk_weights;
    sp.sorted_ids = a->sorted_token_ids;
    sp.expert_ids = a->expert_ids;
    sp.num_post_padded = a->num_tokens_post_padded;
    sp.w13_scale = a->w13_scale;
    sp.w2_scale = a->w2_scale;
    sp.a_sorted = a_sorted;
    sp.as_t = as_t;
    sp.slot_route = slot_route;
    sp.rvalid = rvalid;
    sp.gen = gen;
    sp.slot_w = slot_w;
    sp.wsu = wsu;
    sp.wsd = wsd;
    sp.nblocks = nblocks;
    sp.cap_pad = wl.cap_pad;
    sp.R = static_cast<int>(R);
    sp.top_k = a->top_k;
    sp.block_m = a->block_m;
    sp.E = a->E;
    sp.H = a->H;
    sp.I = a->I;
    sp.routed_scale = a->routed_scale;
    sp.status = a->device_status;
    sp.a_rows = a->sorted_cap;
    sp.check_pow2 = block_scaled ? 1 : 0;
    int64_t sgrid = ceil_div(nblocks * a->block_m, 8);
    if (sgrid > static_cast<int64_t>(dev.sms) * 8) sgrid = static_cast<int64_t>(dev.sms) * 8;
    MOE_CUDA_TRY(launch_pdl(stage_kernel, dim3(static_cast<unsigned>(sgrid)), dim3(256), 0, stream, 1, sp));
    if (ev) MOE_CUDA_TRY(cudaEventRecord(ev[1], stream));

    GemmParams p{};
    p.expert_ids = a->expert_ids;
    p.num_post_padded = a->num_tokens_post_padded;
    p.sorted_ids = a->sorted_token_ids;
    p.status = a->device_status;
    p.nblocks = nblocks;
    p.cap_pad = wl.cap_pad;
    p.R = static_cast<int>(R);
    p.top_k = a->top_k;
    p.block_m = a->block_m;
    p.E = a->E;
    p.I = a->I;
    p.H = a->H;
    p.q_rows = a->sorted_cap;
    p.a_rows = a->sorted_cap;
    p.qbox = qbox;

    GemmParams up = p;
    up.a_scale_t = as_t;
    up.w_scale_st = wsu;
    up.q_inter = q_inter;
    up.s_inter_t = s_inter_t;
    up.dbg_q = a->debug_q_inter;
    up.dbg_s = a->debug_s_inter;
    up.nkb = a->H / 128;
    up.ntiles_n = N / kTileN;
    up.b_rows = N;
    up.a_gather4 = wl.pregather ? 0 : 1;
    if (!wl.pregather) up.a_rows = a->M;
    up.tile_group = 0;
    up.slot_route = slot_route;
    up.gen = gen;
    up.slot_w = slot_w;
    // split K when the tiles cannot fill the GPU (decode): each split streams
    // a share of the weights, the last one to finish applies SwiGLU
    up.splits = 1;
    up.ksplit = up.nkb;
    const int64_t base_tiles = nblocks * up.ntiles_n;
    if (!pair && wl.splitk && base_tiles < dev.sms) {
      int want = static_cast<int>(dev.sms / base_tiles);
      if (want > up.nkb) want = up.nkb;
      if (want > 1) {
        up.ksplit = static_cast<int>(ceil_div(up.nkb, want));
        up.splits = static_cast<int>(ceil_div(up.nkb, up.ksplit));
        up.usum = reinterpret_cast<float*>(ws + wl.usum_off);
        up.ucnt = reinterpret_cast<int32_t*>(ws + wl.ucnt_off);
      }
    }
    const int64_t up_tiles = base_tiles * up.splits;
    if (pair) {
      int64_t clusters = ceil_div(up_tiles, 2);
      if (clusters > pair_clusters) clusters = pair_clusters;
      MOE_CUDA_TRY(launch_pdl(moe_gemm_kernel<true, true>, dim3(static_cast<unsigned>(2 * clusters)),
                              dim3(kNumThreads), smem_bytes<true>(), stream, 2, tm_a, tm_w13, tm_qs, up));
    } else if (block_scaled) {
      const int up_grid = static_cast<int>(up_tiles < dev.sms ? up_tiles : dev.sms);
      MOE_CUDA_TRY(launch_pdl(moe_gemm_kernel<true, false, true>, dim3(up_grid), dim3(kNumThreads),
                              smem_bytes<false>(), stream, 1, tm_a, tm_w13, tm_qs, up));
    } else {
      const int up_grid = static_cast<int>(up_tiles < dev.sms ? up_tiles : dev.sms);
      MOE_CUDA_TRY(launch_pdl(moe_gemm_kernel<true, false>, dim3(up_grid), dim3(kNumThreads), smem_bytes<false>(),
                              stream, 1, tm_a, tm_w13, tm_qs, up));
    }
    if (ev) MOE_CUDA_TRY(cudaEventRecord(ev[2], stream));

    GemmParams dn = p;
    dn.a_scale_t = s_inter_t;
    dn.w_scale_st = wsd;
    dn.slot_route = slot_route;
    dn.slot_w = slot_w;
    dn.y_out = yr;
    dn.nkb = a->I / 128;
    dn.ntiles_n = static_cast<int>(ceil_div(a->H, kTileN));
    dn.b_rows = a->H;
    dn.a_gather4 = 0;
    // Groups of up to 4 n tiles: a plan block's intermediate rows are read by
    // adjacent tiles (one DRAM read per group rather than per n tile: with a
    // single n tile per pass, the pass's weight stream evicts them), while the
    // route reductions of a group touch only its few 256-column stripes of
    // the accumulator, which stay in L2.
    dn.tile_group = 1;
    for (int g = 4; g > 1; --g)
      if (dn.ntiles_n % g == 0) {
        dn.tile_group = g;
        break;
      }
    dn.splits = 1;
    dn.ksplit = dn.nkb;
    const int64_t dn_tiles = nblocks * dn.ntiles_n;
    if (pair) {
      int64_t clusters = ceil_div(dn_tiles, 2);
      if (clusters > pair_clusters) clusters = pair_clusters;
      MOE_CUDA_TRY(launch_pdl(moe_gemm_kernel<false, true>, dim3(static_cast<unsigned>(2 * clusters)),
                              dim3(kNumThreads), smem_bytes<true>(), stream, 2, tm_q, tm_w2, tm_qs, dn));
    } else {
      const int dn_grid = static_cast<int>(dn_tiles < dev.sms ? dn_tiles : dev.sms);
      MOE_CUDA_TRY(launch_pdl(moe_gemm_kernel<false, false>, dim3(dn_grid), dim3(kNumThreads), smem_bytes<false>(),
                              stream, 1, tm_q, tm_w2, tm_qs, dn));
    }
  } else if (ev) {
    MOE_CUDA_TRY(cudaEventRecord(ev[1], stream));
    MOE_CUDA_TRY(cudaEventRecord(ev[2], stream));
  }
  if (ev) MOE_CUDA_TRY(cudaEventRecord(ev[3], stream));

  const int64_t segs = ceil_div(a->H / 8, int64_t(32));
  int64_t fgrid = ceil_div(a->M * segs, int64_t(8));  // a warp per (token, 256-column segment)
  if (fgrid > static_cast<int64_t>(dev.sms) * 32) fgrid = static_cast<int64_t>(dev.sms) * 32;
  MOE_CUDA_TRY(
      launch_pdl(combine_kernel, dim3(static_cast<unsigned>(fgrid)), dim3(256), 0, stream, 1, a->out, yr,
                 static_cast<const uint32_t*>(rvalid), static_cast<const uint32_t*>(gen), a->M, a->H, a->top_k));

  if (ev) MOE_CUDA_TRY(cudaEventRecord(ev[4], stream));
  return MOE_OK;
}

}  // extern "C"

MOE_BOUNDS_TU()
