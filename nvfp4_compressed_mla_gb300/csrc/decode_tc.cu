// decode_tc.cu -- sparse absorbed-MLA decode on the sm_103a tensor cores (tcgen05 + TMEM).
//
// The Prime Inference post, section "Native NVFP4 sparse MLA decode kernel",
// describes a kernel that gathers the compressed rows at the indexer's
// positions, dequantises them on chip, runs FP16 MMAs with FP32
// accumulation, lets separate warp groups dequantise / score / accumulate
// through a three-slot buffer, and merges a query token's partial results
// across a cluster of SMs. This kernel keeps those ideas and reshapes them
// for tcgen05 and its 256 KB of tensor memory per SM.
//
// With 128 heads, one query token's resident state does not fit one SM:
// Q (128 x 576 FP16) and O (128 x 512 FP32, all 512 TMEM columns) together
// exceed both TMEM and shared memory. So each (token, split) unit is a
// 2-CTA cluster that splits the two contractions between two SMs:
//
//   rank 0, "score" CTA: Q lives in TMEM (288 columns, the A operand).
//     Per 64-row tile: S = Q K^T (M=128 heads, N=64 tokens, K=576) into one of
//     two 64-column TMEM score buffers; four softmax warps (one thread per
//     head) read S, keep the running max / sum, and write P (FP16, 128 x 64)
//     straight into the peer's shared memory.
//   rank 1, "output" CTA: O lives in TMEM (512 columns).
//     Per tile: O += P V (M=128, N=2 x 256 latent dims, K=64 tokens), with P
//     and V^T from shared memory. Four correction warps rescale O when the
//     score CTA raises its reference max, forward "P buffer free" back, and
//     write the normalised output at the end.
//
// Both CTAs run the same gather/dequant pipeline on their own copy of the
// rows: a producer warp resolves the top-k slots through the block table
// (-1 and unresolvable slots are skipped: no load is issued) and issues one
// bulk copy (cp.async.bulk) per row into a 3-stage raw ring; eight dequant
// warps expand E2M1 x E4M3 (exact in FP16) into the 128-byte-swizzled
// K-major layout the MMA reads: the score CTA writes K [token][576], the
// output CTA writes V^T [512][token]. One thread issues the MMAs; commits
// signal mbarriers. Softmax uses a lazy reference max: P = 2^(s - m_ref)
// with m_ref raised only when a score exceeds it by more than 8 (P <= 256
// in FP16), so O needs rescaling only on those (rare) tiles.
//
// Every wait is bounded (about a second of clock64 cycles); a wait that
// runs out sets an abort flag, the CTAs unwind, free TMEM, and the unit's
// outputs are written as NaN.
#include <math.h>

#include "decode_common.cuh"

namespace nvfp4_mla {
namespace {

constexpr int kWarps = 14;
constexpr int kThreads = kWarps * 32;
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kDequantWarp0 = 6;
constexpr int kDequantThreads = 256;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kQCol = 0;      // score CTA: Q, 288 columns
constexpr uint32_t kSCol = 384;    // score CTA: score buffers at 384 and 448
constexpr float kTau = 8.0f;       // lazy rescale threshold (log2 units)
constexpr long long kWaitCycles = 1ll << 31;
constexpr uint32_t kIdescQK = (1u << 4) | ((64u >> 3) << 17) | ((128u >> 4) << 24);
constexpr uint32_t kIdescPV = (1u << 4) | ((256u >> 3) << 17) | ((128u >> 4) << 24);

template <int kFmt>
struct TcLayout {
  static constexpr bool kNv = kFmt == NVFP4_MLA_ROW_NVFP4_352;
  static constexpr int kRowBytes = kNv ? kNvfp4Row : kFp8Row;
  static constexpr int kCopyS = kRowBytes;           // score CTA copies whole rows
  static constexpr int kCopyO = kNv ? 288 : 512;     // output CTA: latent part only
  static constexpr int kStages = kNv ? 3 : 2;
  static constexpr int kPad = 16;                    // per 8-row group, against bank conflicts
  static constexpr int kStageS = kTile * kCopyS + 8 * kPad;
  static constexpr int kStageO = kTile * kCopyO + 8 * kPad;
  static constexpr int kKTile = 9 * 8192;            // 64 tokens x 576 FP16, 9 K-blocks of 64
  static constexpr int kRawS = 2 * kKTile;
  static constexpr int kEndS = kRawS + kStages * kStageS;
  static constexpr int kVTile = 64 * 1024;           // 512 dims x 64 tokens FP16
  static constexpr int kPTile = 16 * 1024;           // 128 heads x 64 tokens FP16
  static constexpr int kP = 2 * kVTile;
  static constexpr int kRawO = kP + 2 * kPTile;
  static constexpr int kEndO = kRawO + kStages * kStageO;
  static constexpr int kCtl = ((kEndS > kEndO ? kEndS : kEndO) + 15) / 16 * 16;
  static constexpr int kCtlBytes = 2560;
  static constexpr int kBytes = kCtl + kCtlBytes;
  static_assert(kBytes <= 232448, "shared memory budget");
  static_assert(kStageS % 16 == 0 && kStageO % 16 == 0 && kCopyO % 16 == 0, "bulk copy alignment");
};

// control block (same offset in both CTAs of the cluster)
struct Ctl {
  static constexpr int kRawFull = 0, kRawEmpty = 24, kTileFull = 48, kTileEmpty = 64,
                       kSFull = 80, kSEmpty = 96, kPFull = 112, kPEmpty = 128, kPvDone = 144,
                       kOCorr = 160, kStats = 168, kQReady = 176, kTmem = 192, kAbort = 196,
                       kStageMask = 200, kMaskRing = 224, kFlags = 288, kAlpha = 320,
                       kFinalM = 1344, kFinalL = 1856, kEnd = 2368;
};
static_assert(Ctl::kEnd <= TcLayout<NVFP4_MLA_ROW_NVFP4_352>::kCtlBytes, "control block");

// ------------------------------------------------------------- PTX wrappers
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar)
               : "memory");
}
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n.reg .pred p;\n"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
      "selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint32_t ld_shared_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ void st_shared_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t map_rank(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n"
               "barrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
__device__ __forceinline__ void st_cluster_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                              uint32_t d) {
  asm volatile("st.shared::cluster.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b),
               "r"(c), "r"(d)
               : "memory");
}
__device__ __forceinline__ void st_cluster_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void fence_proxy_async_cta() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_cluster() {
  asm volatile("fence.proxy.async.shared::cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}
__device__ __forceinline__ uint2 ld_shared_v2(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}
__device__ __forceinline__ uint32_t ld_shared_u8(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u8 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

// tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(kTmemCols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr),
               "r"(kTmemCols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D (TMEM) (+)= A (shared, descriptor) * B (shared, descriptor)
__device__ __forceinline__ void mma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D (TMEM) (+)= A (TMEM) * B (shared, descriptor)
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d),
      "r"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::
                   "r"(bar)
               : "memory");
}
#define NVFP4_R8(i) "%" #i ", "
#define NVFP4_TMEM_REGS                                                                          \
  "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, " \
  "%20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}"
#define NVFP4_TMEM_OUTS(r)                                                                      \
  "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),          \
      "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),  \
      "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),            \
      "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),            \
      "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
#define NVFP4_TMEM_INS(r)                                                                        \
  "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),      \
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),        \
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),      \
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),      \
      "r"(r[29]), "r"(r[30]), "r"(r[31])
// 32 consecutive TMEM columns of this thread's lane (32x32b shape)
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 " NVFP4_TMEM_REGS ", [%32];"
               : NVFP4_TMEM_OUTS(r)
               : "r"(taddr)
               : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, "
               "%9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, "
               "%25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
               NVFP4_TMEM_INS(r)
               : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart (stride byte offset), descriptor version 1.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t addr) {
  return static_cast<uint64_t>((addr >> 4) & 0x3FFFu) | (static_cast<uint64_t>(1) << 16) |
         (static_cast<uint64_t>(1024 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
         (static_cast<uint64_t>(2) << 61);
}

// Byte offset of the 16-byte chunk `chunk` (0..7) of row `row` in a 128-byte
// swizzled K-major tile whose rows are 128 bytes (8-row groups of 1024 B).
__device__ __forceinline__ uint32_t sw128_off(uint32_t row, uint32_t chunk) {
  return (row >> 3) * 1024u + (row & 7u) * 128u + ((chunk ^ (row & 7u)) << 4);
}

// Bounded wait; false when it ran out (or another thread aborted already).
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, uint32_t abort_addr) {
  if (mbar_test(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_test(bar, parity)) return true;
    if (ld_shared_u32(abort_addr) != 0) return false;
    if (clock64() - t0 > kWaitCycles) {
      st_shared_u32(abort_addr, 1u);
      return false;
    }
  }
}

// Warp-uniform bounded wait: every lane waits (and so acquires), and the
// warp leaves together, so warp-collective operations after it stay converged.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, uint32_t abort_addr) {
  return __all_sync(0xffffffffu, wait_bar(bar, parity, abort_addr));
}

// Bounded wait that ignores the abort flag: used to drain issued MMAs
// before the tensor memory is freed.
__device__ __forceinline__ void drain_bar(uint32_t bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_test(bar, parity) && clock64() - t0 < kWaitCycles) {
  }
}

__device__ __forceinline__ uint32_t raw_row_off(int t, int copy) {
  return static_cast<uint32_t>(t * copy + (t >> 3) * 16);
}

// ------------------------------------------------------------------ kernel
template <int kFmt>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    decode_tc_kernel(const DecodeParams p) {
  using L = TcLayout<kFmt>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  const uint32_t ctl = sbase + L::kCtl;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_rank();
  const uint32_t peer = rank ^ 1u;

  const int unit = static_cast<int>(blockIdx.x >> 1);
  const int split = unit % p.num_splits;
  const int t = unit / p.num_splits;
  const int tile0 = split * p.tiles_per_split;
  const int n_tiles = min(p.tiles_per_split, p.num_tiles - tile0);

  auto bar = [&](int off, int i) { return ctl + off + 8u * static_cast<uint32_t>(i); };
  const uint32_t abort_addr = ctl + Ctl::kAbort;

  if (tid == 0) {
    for (int s = 0; s < L::kStages; ++s) {
      mbar_init(bar(Ctl::kRawFull, s), 1);
      mbar_init(bar(Ctl::kRawEmpty, s), 8);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(Ctl::kTileFull, s), 8);
      mbar_init(bar(Ctl::kTileEmpty, s), 1);
      mbar_init(bar(Ctl::kSFull, s), 1);
      mbar_init(bar(Ctl::kSEmpty, s), 128);
      mbar_init(bar(Ctl::kPFull, s), 128);
      mbar_init(bar(Ctl::kPEmpty, s), 128);
      mbar_init(bar(Ctl::kPvDone, s), 1);
    }
    mbar_init(bar(Ctl::kOCorr, 0), 128);
    mbar_init(bar(Ctl::kStats, 0), 128);
    mbar_init(bar(Ctl::kQReady, 0), 128);
    st_shared_u32(abort_addr, (sbase & 1023u) != 0 ? 1u : 0u);
    fence_mbar_init();
  }
  if (warp == kMmaWarp) tmem_alloc(ctl + Ctl::kTmem);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync();  // the peer's barriers exist before anyone arrives on them
  const uint32_t tmem = ld_shared_u32(ctl + Ctl::kTmem);

  const int32_t b = __ldg(p.q_seq + t);
  const int32_t len = (b >= 0 && b < p.num_seqs) ? __ldg(p.seq_lens + b) : 0;
  const int32_t* idx_row = p.topk_idx + static_cast<int64_t>(t) * p.topk;
  const int copy = rank == 0 ? L::kCopyS : L::kCopyO;
  const uint32_t raw_base = sbase + (rank == 0 ? L::kRawS : L::kRawO);
  const uint32_t stage_bytes = rank == 0 ? L::kStageS : L::kStageO;

  if (warp == kProducerWarp) {
    // ---------------------------------------------- gather: slots -> rows -> ring
    for (int i = 0; i < n_tiles; ++i) {
      const int s = i % L::kStages;
      const uint32_t k = i / L::kStages;
      if (!warp_wait(bar(Ctl::kRawEmpty, s), (k & 1u) ^ 1u, abort_addr)) break;
      int64_t off[2];
      bool val[2];
      int bad = 0;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int slot = (tile0 + i) * kTile + lane + 32 * j;
        off[j] = -1;
        if (slot < p.topk) {
          const int32_t pos = __ldg(idx_row + slot);
          if (pos != -1) {
            off[j] = resolve_row(b, pos, len, p.block_table, p.num_seqs, p.max_blocks,
                                 p.page_size, p.num_blocks, p.block_stride, L::kRowBytes);
            bad += off[j] < 0;
          }
        }
        val[j] = off[j] >= 0;
      }
      const uint32_t b0 = __ballot_sync(0xffffffffu, val[0]);
      const uint32_t b1 = __ballot_sync(0xffffffffu, val[1]);
      const uint64_t mask = (static_cast<uint64_t>(b1) << 32) | b0;
      if (rank == 0) {
        bad = __reduce_add_sync(0xffffffffu, bad);
        if (lane == 0 && bad > 0 && p.invalid_count != nullptr) atomicAdd(p.invalid_count, bad);
      }
      if (lane == 0) {
        *reinterpret_cast<volatile uint64_t*>(smem + L::kCtl + Ctl::kStageMask + 8 * s) = mask;
        if (rank == 0)
          *reinterpret_cast<volatile uint64_t*>(smem + L::kCtl + Ctl::kMaskRing + 8 * (i & 7)) =
              mask;
        mbar_arrive_tx(bar(Ctl::kRawFull, s), (__popc(b0) + __popc(b1)) * copy);
      }
      __syncwarp();
#pragma unroll
      for (int j = 0; j < 2; ++j)
        if (val[j])
          bulk_g2s(raw_base + s * stage_bytes + raw_row_off(lane + 32 * j, copy),
                   p.cache + off[j], copy, bar(Ctl::kRawFull, s));
    }
  } else if (warp >= kDequantWarp0) {
    // ---------------------------------------------- dequant: raw -> FP16 swizzled tiles
    const int dt = tid - kDequantWarp0 * 32;
    for (int i = 0; i < n_tiles; ++i) {
      const int s = i % L::kStages;
      const uint32_t k = i / L::kStages;
      const int s2 = i & 1;
      const uint32_t k2 = i >> 1;
      if (!warp_wait(bar(Ctl::kRawFull, s), k & 1u, abort_addr)) break;
      if (!warp_wait(bar(Ctl::kTileEmpty, s2), (k2 & 1u) ^ 1u, abort_addr)) break;
      const uint64_t mask =
          *reinterpret_cast<volatile uint64_t*>(smem + L::kCtl + Ctl::kStageMask + 8 * s);
      const uint32_t raw = raw_base + s * stage_bytes;
      if (rank == 0) {
        // K tile [64 tokens][576], 9 K-blocks of 64 dims (8192 B each)
        const uint32_t ktile = sbase + s2 * L::kKTile;
        for (int it = dt; it < kTile * 36; it += kDequantThreads) {
          const int tok = it & 63;
          const int c16 = it >> 6;  // 16-value group 0..35 (32..35: rope)
          uint32_t h[8];
          const uint32_t row = raw + raw_row_off(tok, L::kCopyS);
          if ((mask >> tok) & 1ull) {
            if constexpr (L::kNv) {
              if (c16 < 32) {
                const uint2 pl = ld_shared_v2(row + c16 * 8);
                const uint32_t sc = ld_shared_u8(row + kScaleOff + c16);
                const uint32_t s2h = e4m3x2_to_f16x2(static_cast<uint16_t>(sc | (sc << 8)));
                uint32_t lo[4], hi[4];
                e2m1x8_to_f16x8(pl.x, lo);
                e2m1x8_to_f16x8(pl.y, hi);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                  h[q] = hmul2_u32(lo[q], s2h);
                  h[4 + q] = hmul2_u32(hi[q], s2h);
                }
              } else {
                const uint4 v = ld_shared_v4(row + kRopeOff + (c16 - 32) * 16);
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                  h[2 * q] = e4m3x2_to_f16x2(static_cast<uint16_t>(w[q] & 0xFFFFu));
                  h[2 * q + 1] = e4m3x2_to_f16x2(static_cast<uint16_t>(w[q] >> 16));
                }
              }
            } else {
              const uint4 v = ld_shared_v4(row + c16 * 16);
              const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                h[2 * q] = e4m3x2_to_f16x2(static_cast<uint16_t>(w[q] & 0xFFFFu));
                h[2 * q + 1] = e4m3x2_to_f16x2(static_cast<uint16_t>(w[q] >> 16));
              }
            }
          } else {
#pragma unroll
            for (int q = 0; q < 8; ++q) h[q] = 0u;
          }
          const uint32_t kb = static_cast<uint32_t>(c16 >> 2);
          const uint32_t c0 = static_cast<uint32_t>((c16 & 3) * 2);
          const uint32_t base = ktile + kb * 8192u;
          st_shared_v4(base + sw128_off(tok, c0), h[0], h[1], h[2], h[3]);
          st_shared_v4(base + sw128_off(tok, c0 + 1), h[4], h[5], h[6], h[7]);
        }
      } else {
        // V^T tile [512 dims][64 tokens]: one item = 8 tokens x 16 dims. The
        // transpose happens in registers: each converted f16x2 holds two dims
        // of one token; prmt pairs the same dim of two tokens.
        const uint32_t vtile = sbase + s2 * L::kVTile;
        const int tg = dt & 7;   // token group (8 consecutive tokens)
        const int j = dt >> 3;   // 16-dim group 0..31
        if constexpr (L::kNv) {
          uint32_t pw[8][2], scl[8];
#pragma unroll
          for (int tt = 0; tt < 8; ++tt) {
            const int tok = tg * 8 + tt;
            const uint32_t row = raw + raw_row_off(tok, L::kCopyO);
            const bool ok = (mask >> tok) & 1ull;
            const uint2 pl = ok ? ld_shared_v2(row + j * 8) : make_uint2(0u, 0u);
            pw[tt][0] = pl.x;
            pw[tt][1] = pl.y;
            const uint32_t sc = ok ? ld_shared_u8(row + kScaleOff + j) : 0u;
            scl[tt] = e4m3x2_to_f16x2(static_cast<uint16_t>(sc | (sc << 8)));
          }
#pragma unroll
          for (int wi = 0; wi < 2; ++wi) {
            uint32_t hh[8][4];
#pragma unroll
            for (int tt = 0; tt < 8; ++tt) {
              e2m1x8_to_f16x8(pw[tt][wi], hh[tt]);
#pragma unroll
              for (int q = 0; q < 4; ++q) hh[tt][q] = hmul2_u32(hh[tt][q], scl[tt]);
            }
#pragma unroll
            for (int bq = 0; bq < 4; ++bq) {
              const uint32_t d0 = static_cast<uint32_t>(j * 16 + wi * 8 + 2 * bq);
              st_shared_v4(vtile + sw128_off(d0, tg), prmt(hh[0][bq], hh[1][bq], 0x5410u),
                           prmt(hh[2][bq], hh[3][bq], 0x5410u), prmt(hh[4][bq], hh[5][bq], 0x5410u),
                           prmt(hh[6][bq], hh[7][bq], 0x5410u));
              st_shared_v4(vtile + sw128_off(d0 + 1, tg), prmt(hh[0][bq], hh[1][bq], 0x7632u),
                           prmt(hh[2][bq], hh[3][bq], 0x7632u), prmt(hh[4][bq], hh[5][bq], 0x7632u),
                           prmt(hh[6][bq], hh[7][bq], 0x7632u));
            }
          }
        } else {
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            uint32_t ww[8][2];
#pragma unroll
            for (int tt = 0; tt < 8; ++tt) {
              const int tok = tg * 8 + tt;
              const uint32_t row = raw + raw_row_off(tok, L::kCopyO);
              const bool ok = (mask >> tok) & 1ull;
              const uint2 v = ok ? ld_shared_v2(row + j * 16 + half * 8) : make_uint2(0u, 0u);
              ww[tt][0] = v.x;
              ww[tt][1] = v.y;
            }
#pragma unroll
            for (int pi = 0; pi < 4; ++pi) {  // byte pair pi -> dims 2pi, 2pi+1 of this half
              uint32_t f[8];
#pragma unroll
              for (int tt = 0; tt < 8; ++tt)
                f[tt] = e4m3x2_to_f16x2(
                    static_cast<uint16_t>((ww[tt][pi >> 1] >> (16 * (pi & 1))) & 0xFFFFu));
              const uint32_t d0 = static_cast<uint32_t>(j * 16 + half * 8 + 2 * pi);
              st_shared_v4(vtile + sw128_off(d0, tg), prmt(f[0], f[1], 0x5410u),
                           prmt(f[2], f[3], 0x5410u), prmt(f[4], f[5], 0x5410u),
                           prmt(f[6], f[7], 0x5410u));
              st_shared_v4(vtile + sw128_off(d0 + 1, tg), prmt(f[0], f[1], 0x7632u),
                           prmt(f[2], f[3], 0x7632u), prmt(f[4], f[5], 0x7632u),
                           prmt(f[6], f[7], 0x7632u));
            }
          }
        }
      }
      fence_proxy_async_cta();  // generic-proxy stores -> visible to the tensor core
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(bar(Ctl::kTileFull, s2));
        mbar_arrive(bar(Ctl::kRawEmpty, s));
      }
    }
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------- MMA issue (one thread)
    if (lane == 0) {
      int issued = 0;
      if (rank == 0) {
        if (wait_bar(bar(Ctl::kQReady, 0), 0, abort_addr)) {
          for (int i = 0; i < n_tiles; ++i) {
            const int s2 = i & 1;
            const uint32_t k2 = i >> 1;
            if (!wait_bar(bar(Ctl::kTileFull, s2), k2 & 1u, abort_addr)) break;
            if (!wait_bar(bar(Ctl::kSEmpty, s2), (k2 & 1u) ^ 1u, abort_addr)) break;
            tc_fence_after();
            const uint32_t ktile = sbase + s2 * L::kKTile;
            const uint32_t dcol = tmem + kSCol + 64u * s2;
#pragma unroll 4
            for (int kk = 0; kk < 36; ++kk) {
              const uint64_t bdesc = sw128_desc(ktile + (kk >> 2) * 8192u + (kk & 3) * 32u);
              mma_ts(dcol, tmem + kQCol + 8u * kk, bdesc, kIdescQK, kk > 0 ? 1u : 0u);
            }
            mma_commit(bar(Ctl::kTileEmpty, s2));
            mma_commit(bar(Ctl::kSFull, s2));
            issued = i + 1;
          }
        }
      } else {
        uint32_t n_corr = 0;
        for (int i = 0; i < n_tiles; ++i) {
          const int s2 = i & 1;
          const uint32_t k2 = i >> 1;
          if (!wait_bar(bar(Ctl::kTileFull, s2), k2 & 1u, abort_addr)) break;
          if (!wait_bar(bar(Ctl::kPFull, s2), k2 & 1u, abort_addr)) break;
          const uint4 fl = ld_shared_v4(ctl + Ctl::kFlags + 16 * s2);
          if ((fl.x | fl.y | fl.z | fl.w) != 0u) {
            if (!wait_bar(bar(Ctl::kOCorr, 0), n_corr & 1u, abort_addr)) break;
            ++n_corr;
          }
          tc_fence_after();
          fence_proxy_async_cta();
          const uint32_t vtile = sbase + s2 * L::kVTile;
          const uint32_t ptile = sbase + L::kP + s2 * L::kPTile;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t adesc = sw128_desc(ptile + kk * 32u);
#pragma unroll
            for (int nh = 0; nh < 2; ++nh) {
              const uint64_t bdesc = sw128_desc(vtile + nh * 32768u + kk * 32u);
              mma_ss(tmem + 256u * nh, adesc, bdesc, kIdescPV, (i > 0 || kk > 0) ? 1u : 0u);
            }
          }
          mma_commit(bar(Ctl::kTileEmpty, s2));
          mma_commit(bar(Ctl::kPvDone, s2));
          issued = i + 1;
        }
      }
      if (issued > 0) {  // the last commit completes once every MMA issued here has
        const int last = issued - 1;
        drain_bar(bar(Ctl::kTileEmpty, last & 1), (static_cast<uint32_t>(last) >> 1) & 1u);
      }
    }
  } else if (rank == 0) {
    // ---------------------------------------------- score CTA: Q -> TMEM, then softmax
    const int h = warp * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    {
      const bool live = h < p.num_heads;
      const int64_t qh = static_cast<int64_t>(t) * p.num_heads + h;
#pragma unroll 1
      for (int c = 0; c < 9; ++c) {
        uint32_t r[32];
        const float m = c < 8 ? p.q_lat_mult : p.q_rope_mult;
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          uint4 x = make_uint4(0u, 0u, 0u, 0u);
          if (live)
            x = c < 8 ? ld_nc_v4(p.q_lat + qh * kLatent + c * 64 + v * 8)
                      : ld_nc_v4(p.q_rope + qh * kRope + v * 8);
          r[4 * v + 0] = pack_f16x2(bf16_lo(x.x) * m, bf16_hi(x.x) * m);
          r[4 * v + 1] = pack_f16x2(bf16_lo(x.y) * m, bf16_hi(x.y) * m);
          r[4 * v + 2] = pack_f16x2(bf16_lo(x.z) * m, bf16_hi(x.z) * m);
          r[4 * v + 3] = pack_f16x2(bf16_lo(x.w) * m, bf16_hi(x.w) * m);
        }
        tmem_st32(tmem + lane_base + kQCol + 32u * c, r);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(Ctl::kQReady, 0));
    }
    const uint32_t peer_p = map_rank(sbase + L::kP, peer);
    const uint32_t peer_ctl = map_rank(ctl, peer);
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    for (int i = 0; i < n_tiles; ++i) {
      const int s2 = i & 1;
      const uint32_t k2 = i >> 1;
      if (!warp_wait(bar(Ctl::kSFull, s2), k2 & 1u, abort_addr)) { ok = false; break; }
      tc_fence_after();
      const uint64_t mask =
          *reinterpret_cast<volatile uint64_t*>(smem + L::kCtl + Ctl::kMaskRing + 8 * (i & 7));
      uint32_t sa[32], sb[32];
      tmem_ld32(tmem + lane_base + kSCol + 64u * s2, sa);
      tmem_ld32(tmem + lane_base + kSCol + 64u * s2 + 32u, sb);
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(bar(Ctl::kSEmpty, s2));
      float mx = -INFINITY;
#pragma unroll
      for (int q = 0; q < 32; ++q) {
        const float v0 = ((mask >> q) & 1ull) ? __uint_as_float(sa[q]) * p.score_scale : -INFINITY;
        const float v1 =
            ((mask >> (32 + q)) & 1ull) ? __uint_as_float(sb[q]) * p.score_scale : -INFINITY;
        sa[q] = __float_as_uint(v0);
        sb[q] = __float_as_uint(v1);
        mx = fmaxf(mx, fmaxf(v0, v1));
      }
      float alpha = 1.f;
      bool resc = false;
      if (mx > m_ref + kTau) {  // also the first valid score (m_ref = -inf)
        alpha = m_ref == -INFINITY ? 0.f : ex2(m_ref - mx);
        m_ref = mx;
        l *= alpha;
        resc = true;
      }
      uint32_t pk[32];
      float sum = 0.f;
#pragma unroll
      for (int q = 0; q < 32; ++q) {
        const uint32_t* src = q < 16 ? sa : sb;
        const int qq = (q & 15) * 2;
        const float p0 = m_ref == -INFINITY ? 0.f : ex2(__uint_as_float(src[qq]) - m_ref);
        const float p1 = m_ref == -INFINITY ? 0.f : ex2(__uint_as_float(src[qq + 1]) - m_ref);
        pk[q] = pack_f16x2(p0, p1);
        sum += f16_bits_to_f32(static_cast<uint16_t>(pk[q] & 0xFFFFu)) +
               f16_bits_to_f32(static_cast<uint16_t>(pk[q] >> 16));
      }
      l += sum;
      // P buffer s2 of the peer is free once its PV of tile i-2 completed
      if (!warp_wait(bar(Ctl::kPEmpty, s2), (k2 & 1u) ^ 1u, abort_addr)) { ok = false; break; }
      const uint32_t prow = peer_p + s2 * L::kPTile;
#pragma unroll
      for (int c = 0; c < 8; ++c)
        st_cluster_v4(prow + sw128_off(h, c), pk[4 * c], pk[4 * c + 1], pk[4 * c + 2],
                      pk[4 * c + 3]);
      st_cluster_u32(peer_ctl + Ctl::kAlpha + 4 * (s2 * 128 + h), __float_as_uint(alpha));
      const bool warp_resc = __any_sync(0xffffffffu, resc && i > 0);
      if (lane == 0)
        st_cluster_u32(peer_ctl + Ctl::kFlags + 16 * s2 + 4 * warp, warp_resc ? 1u : 0u);
      fence_proxy_async_cluster();
      mbar_arrive_cluster(peer_ctl + Ctl::kPFull + 8 * s2);
    }
    if (ok) {
      st_cluster_u32(peer_ctl + Ctl::kFinalM + 4 * h, __float_as_uint(m_ref));
      st_cluster_u32(peer_ctl + Ctl::kFinalL + 4 * h, __float_as_uint(l));
      mbar_arrive_cluster(peer_ctl + Ctl::kStats);
    }
  } else {
    // ---------------------------------------------- output CTA: corrections + epilogue
    const int h = warp * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t peer_ctl = map_rank(ctl, peer);
    uint32_t n_corr = 0;
    bool ok = true;
    for (int i = 0; i < n_tiles; ++i) {
      const int s2 = i & 1;
      const uint32_t k2 = i >> 1;
      if (!warp_wait(bar(Ctl::kPvDone, s2), k2 & 1u, abort_addr)) { ok = false; break; }
      tc_fence_after();
      // every correction thread read this slot's flags/alpha already (tile i, in
      // the previous iteration): the score CTA may now refill the slot
      mbar_arrive_cluster(peer_ctl + Ctl::kPEmpty + 8 * s2);
      if (i + 1 < n_tiles) {
        const int n2 = (i + 1) & 1;
        const uint32_t nk2 = (i + 1) >> 1;
        if (!warp_wait(bar(Ctl::kPFull, n2), nk2 & 1u, abort_addr)) { ok = false; break; }
        const uint4 fl = ld_shared_v4(ctl + Ctl::kFlags + 16 * n2);
        if ((fl.x | fl.y | fl.z | fl.w) != 0u) {
          const float alpha =
              *reinterpret_cast<volatile float*>(smem + L::kCtl + Ctl::kAlpha + 4 * (n2 * 128 + h));
#pragma unroll 1
          for (int c = 0; c < 16; ++c) {
            uint32_t r[32];
            tmem_ld32(tmem + lane_base + 32u * c, r);
            tmem_ld_wait();
#pragma unroll
            for (int q = 0; q < 32; ++q) r[q] = __float_as_uint(__uint_as_float(r[q]) * alpha);
            tmem_st32(tmem + lane_base + 32u * c, r);
          }
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(bar(Ctl::kOCorr, 0));
          ++n_corr;
        }
      }
    }
    float m_fin = NAN, l_fin = 0.f;
    ok = __all_sync(0xffffffffu, ok);
    if (ok && warp_wait(bar(Ctl::kStats, 0), 0, abort_addr)) {
      m_fin = *reinterpret_cast<volatile float*>(smem + L::kCtl + Ctl::kFinalM + 4 * h);
      l_fin = *reinterpret_cast<volatile float*>(smem + L::kCtl + Ctl::kFinalL + 4 * h);
    } else {
      ok = false;
    }
    tc_fence_after();
    {
      const bool live = h < p.num_heads;  // TMEM loads are warp-wide; only stores are per lane
      const float inv = !ok ? NAN : (l_fin > 0.f ? 1.f / l_fin : 0.f);
      const float lse_nat = !ok ? NAN : (l_fin > 0.f ? (m_fin + lg2(l_fin)) * kLn2 : -INFINITY);
      const int64_t qh = static_cast<int64_t>(t) * p.num_heads + h;
      const bool single = p.num_splits == 1;
      const float sc = single ? inv * p.out_mult : inv;
      const int64_t part = (static_cast<int64_t>(t) * p.num_splits + split) * p.num_heads + h;
#pragma unroll 1
      for (int c = 0; c < 16; ++c) {
        uint32_t r[32];
        if (ok) {
          tmem_ld32(tmem + lane_base + 32u * c, r);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int q = 0; q < 32; ++q) r[q] = 0u;
        }
        if (!live) continue;
        float v[32];
#pragma unroll
        for (int q = 0; q < 32; ++q) v[q] = __uint_as_float(r[q]) * sc;
        if (single && !p.out_fp32) {
          uint4* dst =
              reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + qh * kLatent + c * 32);
#pragma unroll
          for (int q = 0; q < 4; ++q)
            dst[q] = make_uint4(pack_bf16x2(v[8 * q], v[8 * q + 1]),
                                pack_bf16x2(v[8 * q + 2], v[8 * q + 3]),
                                pack_bf16x2(v[8 * q + 4], v[8 * q + 5]),
                                pack_bf16x2(v[8 * q + 6], v[8 * q + 7]));
        } else {
          float* dst = single ? static_cast<float*>(p.out) + qh * kLatent + c * 32
                              : p.ws + part * kLatent + c * 32;
#pragma unroll
          for (int q = 0; q < 8; ++q)
            reinterpret_cast<float4*>(dst)[q] =
                make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        }
      }
      if (live) {
        if (single) {
          if (p.lse != nullptr) p.lse[qh] = lse_nat;
        } else {
          p.ws[static_cast<int64_t>(p.num_q) * p.num_splits * p.num_heads * kLatent + part] =
              lse_nat;
        }
      }
    }
  }

  // ---------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem);
  }
  cluster_sync();  // no peer access to this CTA's shared memory after this point
}

template <int kFmt>
int32_t launch_fmt(const DecodeParams& p, cudaStream_t stream) {
  constexpr int smem = TcLayout<kFmt>::kBytes;
  cudaFuncSetAttribute(decode_tc_kernel<kFmt>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  const int64_t ctas = 2ll * p.num_q * p.num_splits;
  if (ctas > 0x7FFFFFFF) return NVFP4_MLA_ERR_SHAPE;
  decode_tc_kernel<kFmt><<<static_cast<unsigned>(ctas), kThreads, smem, stream>>>(p);
  return launch_status();
}

}  // namespace

int32_t launch_decode_tc(const DecodeParams& p, int row_format, cudaStream_t stream) {
  if (row_format == NVFP4_MLA_ROW_FP8_576) return launch_fmt<NVFP4_MLA_ROW_FP8_576>(p, stream);
  return launch_fmt<NVFP4_MLA_ROW_NVFP4_352>(p, stream);
}

}  // namespace nvfp4_mla
