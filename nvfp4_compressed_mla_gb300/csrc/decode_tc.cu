// decode_tc.cu -- sparse absorbed-MLA decode on the sm_103a tensor cores (tcgen05 + TMEM).
//
// The Prime Inference post, section "Native NVFP4 sparse MLA decode kernel",
// describes a kernel that gathers the compressed rows at the indexer's
// positions, dequantises them on chip, runs FP16 MMAs with FP32
// accumulation, lets separate warp groups dequantise / score / accumulate
// through a multi-slot buffer, and merges a query token's partial results
// across a cluster of SMs. This kernel keeps those ideas and reshapes them
// for tcgen05 and its 512 columns of tensor memory per SM.
//
// With 128 heads, one query token's resident state does not fit one SM:
// Q (128 x 576 FP16) and O (128 x 512 FP32, all 512 TMEM columns) together
// exceed both TMEM and shared memory. Each (token, split) unit is a 2-CTA
// cluster that splits the two contractions between two SMs:
//
//   rank 0, "score" CTA: Q_latent lives in TMEM (256 columns, the MMA's A
//     operand) and Q_rope in shared memory. Per 128-row tile, S = Q K^T
//     (M=128 heads, N=128 rows) accumulates into one of two 128-column TMEM
//     buffers, fed by 64-dim chunks of K (128 rows x 64 dims FP16) that the
//     dequant warps write into a 4-slot ring: 8 latent chunks with A from
//     TMEM, then the rope chunk with A from shared memory. N=128 keeps each
//     MMA well above the tensor core's per-instruction floor, and the chunk
//     ring bounds shared memory independently of the tile width.
//     Four softmax warps (one thread per head) read S in two 64-row halves,
//     keep a lazy reference max and the running sum, stage P (FP16) with the
//     rescale factors locally and bulk-copy them into the peer's memory.
//   rank 1, "output" CTA: O lives in TMEM (512 columns). Per 64-row
//     sub-tile: O += P V (M=128, N=2 x 256 latent dims, K=64 rows), P and V^T
//     from shared memory. Four correction warps rescale O when the score CTA
//     raised its reference max, hand P buffers back, and write the
//     normalised output at the end.
//
// Both CTAs gather their own copy of the rows: a producer warp resolves
// top-k slots through the block table (-1 and unresolvable slots issue no
// load), batching the index and block-table loads four stages ahead, and
// publishes per 64-slot stage the rows' byte offsets and a live-row mask.
// Two copy warps gather the live rows with tile::gather4 tensor copies (four
// rows per copy; one bulk copy per row when the page stride is not a whole
// number of rows) into rows padded to an odd number of 16-byte units, so
// eight consecutive rows hit distinct bank groups. Eight dequant warps then
// expand E2M1 x E4M3 (exact in FP16) into the 128-byte-swizzled layouts the
// MMAs read (K-major K chunks in the score CTA, MN-major V slots in the
// output CTA). One thread issues the MMAs; commits signal mbarriers. The
// MMA warp shares its SM sub-partition with the two copy warps rather than
// with dequant warps. Softmax: P = 2^(s - m_ref) with m_ref raised only when
// a score exceeds it by more than 8 (so P <= 256 in FP16) and O rescaled
// only on those (rare) tiles.
//
// Every wait is bounded (about a second of clock64 cycles); a wait that
// runs out sets an abort flag, the roles unwind together, tensor memory is
// freed, and the unit's outputs are written as NaN.
#include <cuda.h>
#include <math.h>
#include <string.h>

#include <mutex>

#include "decode_common.cuh"

namespace nvfp4_mla {
namespace {

constexpr int kSub = 64;             // rows per gather stage / P sub-tile
constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
// Gather copies: warps 9 and 13; dequant: warps 6, 7, 8, 10, 11, 12, 14, 15.
// Warp w runs on SM sub-partition w % 4; sub-partition 1 holds the MMA warp
// with the two light copy warps (and one softmax / correction warp) so that
// the single MMA-issuing thread does not compete with dequant warps.
constexpr int kCopyWarpA = 9, kCopyWarpB = 13;
__device__ __forceinline__ bool is_copy_warp(int w) { return w == kCopyWarpA || w == kCopyWarpB; }
__device__ __forceinline__ int dequant_index(int w) {  // 0..7 for the dequant warps
  return w - 6 - (w > kCopyWarpA ? 1 : 0) - (w > kCopyWarpB ? 1 : 0);
}
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSCol = 256;      // score CTA: S buffers at columns 256 and 384
constexpr int kChunkSlots = 4;
constexpr int kChunksPerTile = 9;    // 8 latent + 1 rope
constexpr float kTau = 8.0f;         // lazy rescale threshold (log2 units)
constexpr long long kWaitCycles = 1ll << 31;
constexpr uint32_t kIdescQK = (1u << 4) | ((128u >> 3) << 17) | ((128u >> 4) << 24);
// P V: B (= V, rows x dims) is read MN-major (dims contiguous): bit 16
constexpr uint32_t kIdescPV = (1u << 4) | (1u << 16) | ((256u >> 3) << 17) | ((128u >> 4) << 24);
constexpr uint32_t kAFBytes = 528;   // per P buffer: 128 fp32 rescale factors + 4 warp flags

template <int kFmt>
struct TcLayout {
  static constexpr bool kNv = kFmt == NVFP4_MLA_ROW_NVFP4_352;
  static constexpr int kRowBytes = kNv ? kNvfp4Row : kFp8Row;
  // Gathered rows: the score CTA keeps whole rows, the output CTA the latent
  // part (plus 16 bytes); both padded to an odd number of 16-byte units so
  // eight consecutive rows hit distinct bank groups. Tensor copies write
  // groups of four rows; groups start 128-byte aligned.
  static constexpr int kElem = kNv ? 2 : 4;                 // tensor-map element bytes
  static constexpr int kRowElems = kRowBytes / kElem;       // 176 / 144
  static constexpr int kRowS = kNv ? 368 : 592;             // whole row + 16 zero-filled bytes
  static constexpr int kRowO = kNv ? 304 : 528;             // latent (+ 16 bytes of the rope)
  static constexpr int kCopyS = kRowBytes;                  // per-row copies (fallback)
  static constexpr int kCopyO = kNv ? 288 : 512;
  static constexpr int kGroupS = (4 * kRowS + 127) / 128 * 128;  // 1536 / 2432
  static constexpr int kGroupO = (4 * kRowO + 127) / 128 * 128;  // 1280 / 2176
  static constexpr int kStageS = 16 * kGroupS;
  static constexpr int kStageO = 16 * kGroupO;
  static constexpr int kStagesS = kNv ? 4 : 2;
  static constexpr int kStagesO = kNv ? 3 : 2;
  static constexpr int kOffsSlots = kNv ? 8 : 6;  // resolved stages: 64 byte offsets + live mask
  static constexpr int kOffsSlot = kSub * 8 + 8;
  static constexpr int kOffsBytes = kOffsSlots * kOffsSlot;
  // score CTA
  static constexpr int kChunk = 16384;            // 128 rows x 64 dims FP16
  static constexpr int kQRope = kChunkSlots * kChunk;
  static constexpr int kPStage = kQRope + 16384;  // 2 x [P 16 KB][rescale + flags]
  static constexpr int kPStageStride = 17408;
  static constexpr int kRawS = kPStage + 2 * kPStageStride;
  static constexpr int kOffsS = kRawS + kStagesS * kStageS;
  static constexpr int kEndS = kOffsS + kOffsBytes;
  static constexpr int kQStage = 0;               // start-up: Q (bf16) staged over the above
  static constexpr int kQPitch = kLatent * 2 + 16; // latent rows padded: conflict-free row reads
  static constexpr int kQRopeStage = 128 * kQPitch;
  static constexpr int kQStageBytes = kQRopeStage + 128 * kRope * 2;
  // output CTA
  static constexpr int kVSlot = 32 * 1024;        // 32 rows x 512 dims FP16 (MN-major)
  static constexpr int kVSlots = 3;
  static constexpr int kPTile = 16 * 1024;        // 128 heads x 64 rows FP16
  static constexpr int kP = kVSlots * kVSlot;
  static constexpr int kRawO = kP + 2 * kPTile;
  static constexpr int kOffsO = kRawO + kStagesO * kStageO;
  static constexpr int kEndO = kOffsO + kOffsBytes;
  static constexpr int kCtl = ((kEndS > kEndO ? kEndS : kEndO) + 15) / 16 * 16;
  static constexpr int kCtlBytes = 2768;
  static constexpr int kBytes = kCtl + kCtlBytes;
  static_assert(kBytes <= 232448, "shared memory budget");
  static_assert(kQStageBytes <= kRawS + kStagesS * kStageS, "Q staging fits the score CTA's buffers");
  static_assert(kStageS % 128 == 0 && kStageO % 128 == 0 && kP % 1024 == 0, "alignment");
  static_assert(kRawS % 128 == 0 && kRawO % 128 == 0, "tensor-copy destinations");
  static_assert(128 * (1024 + 16) <= kRawO + kStagesO * kStageO, "epilogue staging fits");
};

// control block: same offset in both CTAs of the cluster
struct Ctl {
  static constexpr int kRawFull = 0, kRawEmpty = 32, kChunkFull = 64, kChunkEmpty = 96,
                       kVtFull = 128, kVtEmpty = 152, kSFull = 176, kSEmpty = 192, kPFull = 208,
                       kPEmpty = 224, kPvDone = 240, kOCorr = 256, kStats = 264, kQReady = 272,
                       kQFull = 280, kOffsFull = 288, kOffsEmpty = 352, kTmem = 416,
                       kAbort = 420, kMaskRing = 424, kAF = 688, kFinalM = 1744, kFinalL = 2256,
                       kEnd = 2768;
};
static_assert(Ctl::kEnd <= TcLayout<NVFP4_MLA_ROW_NVFP4_352>::kCtlBytes, "control block");
static_assert(Ctl::kAF + 2 * kAFBytes <= Ctl::kFinalM, "rescale/flag slots");

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
__device__ __forceinline__ void mbar_arrive_cluster_relaxed(uint32_t cluster_bar) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar)
               : "memory");
}
// Phase test. Barriers that only this CTA's threads, copies and MMAs arrive
// on are waited with CTA-scope acquire; cluster scope (a costlier fence) is
// kept for the few that the peer CTA arrives on.
template <bool kCluster = false>
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  if constexpr (kCluster)
    asm volatile(
        "{\n.reg .pred p;\n"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
        "selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
  else
    asm volatile(
        "{\n.reg .pred p;\n"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n"
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
__device__ __forceinline__ void st_cluster_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void fence_proxy_async_cta() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
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

// Relaxed: the bytes that complete the phase arrive by the bulk copy's own
// complete_tx, so no release ordering is needed (a release.cluster arrive
// costs a cluster-wide fence of several hundred cycles).
__device__ __forceinline__ void mbar_arrive_tx_cluster(uint32_t cluster_bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.relaxed.cluster.shared::cluster.b64 _, [%0], %1;" ::
                   "r"(cluster_bar),
               "r"(bytes)
               : "memory");
}
// shared (this CTA) -> shared (cluster peer), completion counted on the peer's mbarrier
__device__ __forceinline__ void bulk_s2s(uint32_t dst_cluster, uint32_t src, uint32_t bytes,
                                         uint32_t bar_cluster) {
  asm volatile(
      "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst_cluster),
      "r"(src), "r"(bytes), "r"(bar_cluster)
      : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
template <int kPending>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(kPending) : "memory");
}
// Barrier 1 over the 128 threads of warps 0-3, returning the AND of `v` over them.
__device__ __forceinline__ bool group_and(bool v) {
  uint32_t r;
  asm volatile(
      "{\n.reg .pred p, q;\nsetp.ne.u32 p, %1, 0;\n"
      "bar.red.and.pred q, 1, 128, p;\nselp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"(v ? 1u : 0u)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void group_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// four rows (y0..y3) of a 2-D tensor map, one box each, into consecutive boxes at dst
__device__ __forceinline__ void gather4(uint32_t dst, const CUtensorMap* tm, int32_t y0, int32_t y1,
                                        int32_t y2, int32_t y3, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(0), "r"(y0), "r"(y1), "r"(y2), "r"(y3), "r"(bar)
      : "memory");
}
__device__ __forceinline__ uint64_t ld_shared_u64(uint32_t addr) {
  uint64_t v;
  asm volatile("ld.shared.u64 %0, [%1];" : "=l"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ void st_shared_u64(uint32_t addr, uint64_t v) {
  asm volatile("st.shared.u64 [%0], %1;" ::"r"(addr), "l"(v) : "memory");
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart (stride byte offset), descriptor version 1.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t addr) {
  return static_cast<uint64_t>((addr >> 4) & 0x3FFFu) | (static_cast<uint64_t>(1) << 16) |
         (static_cast<uint64_t>(1024 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
         (static_cast<uint64_t>(2) << 61);
}

// The same for an MN-major operand whose 64-element blocks along N are 4096
// bytes apart (leading byte offset) and whose 8-row groups along K are 1024
// bytes apart (stride byte offset).
__device__ __forceinline__ uint64_t sw128_desc_mn(uint32_t addr) {
  return static_cast<uint64_t>((addr >> 4) & 0x3FFFu) | (static_cast<uint64_t>(4096 >> 4) << 16) |
         (static_cast<uint64_t>(1024 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
         (static_cast<uint64_t>(2) << 61);
}

// Byte offset of 16-byte chunk `chunk` (0..7) of row `row` in a 128-byte
// swizzled K-major tile with 128-byte rows (8-row groups of 1024 bytes).
__device__ __forceinline__ uint32_t sw128_off(uint32_t row, uint32_t chunk) {
  return (row >> 3) * 1024u + (row & 7u) * 128u + ((chunk ^ (row & 7u)) << 4);
}

// Bounded wait; false when it ran out (or another thread of the CTA aborted).
// try_wait with a suspend-time hint: a waiting thread sleeps until the phase
// completes (or the hint expires) instead of spinning.
constexpr uint32_t kSuspendNs = 20000;
template <bool kCluster>
__device__ __forceinline__ bool mbar_wait_suspend(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  if constexpr (kCluster)
    asm volatile(
        "{\n.reg .pred p;\n"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n"
        "selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(kSuspendNs)
        : "memory");
  else
    asm volatile(
        "{\n.reg .pred p;\n"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n"
        "selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(kSuspendNs)
        : "memory");
  return ok != 0;
}
template <bool kCluster = false>
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, uint32_t abort_addr) {
  if (mbar_test<kCluster>(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_wait_suspend<kCluster>(bar, parity)) return true;
    if (ld_shared_u32(abort_addr) != 0) return false;
    if (clock64() - t0 > kWaitCycles) {
      st_shared_u32(abort_addr, 1u);
      return false;
    }
  }
}

// Warp-uniform bounded wait: every lane waits (and so acquires) and the
// warp leaves together, so warp-collective operations after it stay converged.
template <bool kCluster = false>
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, uint32_t abort_addr) {
  return __all_sync(0xffffffffu, wait_bar<kCluster>(bar, parity, abort_addr));
}

// Bounded wait that ignores the abort flag: drains issued MMAs before the
// tensor memory is freed.
__device__ __forceinline__ void drain_bar(uint32_t bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_test(bar, parity) && clock64() - t0 < kWaitCycles) {
  }
}


// Packed fp32 pairs (sm_100 family): one instruction does two lanes' worth
// of fma / add; three-input max.
__device__ __forceinline__ uint64_t f32x2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f32x2_split(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t add_f32x2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// FP16x2 of two fp32 p values and the conversions of the Q rows.
__device__ __forceinline__ uint4 bf16x8_to_f16x8(uint4 x, float m) {
  return make_uint4(pack_f16x2(bf16_lo(x.x) * m, bf16_hi(x.x) * m),
                    pack_f16x2(bf16_lo(x.y) * m, bf16_hi(x.y) * m),
                    pack_f16x2(bf16_lo(x.z) * m, bf16_hi(x.z) * m),
                    pack_f16x2(bf16_lo(x.w) * m, bf16_hi(x.w) * m));
}

// E4M3 bytes (16) -> FP16 (16 values = two 16-byte chunks)
__device__ __forceinline__ void e4m3x16_to_f16(uint4 v, uint32_t (&h)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    h[2 * q] = e4m3x2_to_f16x2(static_cast<uint16_t>(w[q] & 0xFFFFu));
    h[2 * q + 1] = e4m3x2_to_f16x2(static_cast<uint16_t>(w[q] >> 16));
  }
}

// ------------------------------------------------------------------ kernel
template <int kFmt>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    decode_tc_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap tm_s,
                     const __grid_constant__ CUtensorMap tm_o) {
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
  const int n_sub = 2 * n_tiles;

  // The resolve warp's first global loads (sequence, length, the first four
  // stages' top-k slots) go out before the set-up, so their latency overlaps it.
  const int32_t b = __ldg(p.q_seq + t);
  const int32_t len = (b >= 0 && b < p.num_seqs) ? __ldg(p.seq_lens + b) : 0;
  const int32_t* idx_row = p.topk_idx + static_cast<int64_t>(t) * p.topk;
  auto load_pos = [&](int u, int32_t (&pos)[2]) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int slot = tile0 * kTile + u * kSub + lane + 32 * j;
      pos[j] = (u < n_sub && slot < p.topk) ? __ldg(idx_row + slot) : -1;
    }
  };
  int32_t posa[4][2];
  if (warp == kProducerWarp) {
#pragma unroll
    for (int k = 0; k < 4; ++k) load_pos(k, posa[k]);
  }

  auto bar = [&](int off, int i) { return ctl + off + 8u * static_cast<uint32_t>(i); };
  const uint32_t abort_addr = ctl + Ctl::kAbort;
  const int stages = rank == 0 ? L::kStagesS : L::kStagesO;

  if (tid == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(bar(Ctl::kRawFull, s), 1);  // armed with the stage's bytes, then bulk copies
      mbar_init(bar(Ctl::kRawEmpty, s), 8);
    }
    for (int s = 0; s < L::kOffsSlots; ++s) {
      mbar_init(bar(Ctl::kOffsFull, s), 1);
      mbar_init(bar(Ctl::kOffsEmpty, s), 2);  // one arrival per copy-issuing warp
    }
    for (int s = 0; s < kChunkSlots; ++s) {
      mbar_init(bar(Ctl::kChunkFull, s), 8);
      mbar_init(bar(Ctl::kChunkEmpty, s), 1);
    }
    for (int s = 0; s < L::kVSlots; ++s) {
      mbar_init(bar(Ctl::kVtFull, s), 8);
      mbar_init(bar(Ctl::kVtEmpty, s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(Ctl::kSFull, s), 1);
      mbar_init(bar(Ctl::kSEmpty, s), 128);
      mbar_init(bar(Ctl::kPFull, s), 1);
      mbar_init(bar(Ctl::kPEmpty, s), 4);
      mbar_init(bar(Ctl::kPvDone, s), 1);
    }
    mbar_init(bar(Ctl::kOCorr, 0), 128);
    mbar_init(bar(Ctl::kStats, 0), 128);
    mbar_init(bar(Ctl::kQReady, 0), 128);
    mbar_init(bar(Ctl::kQFull, 0), 1);
    st_shared_u32(abort_addr, (sbase & 1023u) != 0 ? 1u : 0u);
    fence_mbar_init();
  }
  if (warp == kMmaWarp) tmem_alloc(ctl + Ctl::kTmem);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync();  // the peer's barriers exist before anyone arrives on them
  const uint32_t tmem = ld_shared_u32(ctl + Ctl::kTmem);
  if (tmem != 0u && tid == 0) st_shared_u32(abort_addr, 1u);  // MMA operands assume base 0

  if (rank == 0) {
    // Q of this token, issued first and spread over the 13 warps other than
    // the resolve and copy warps (a copy instruction stalls its warp for a
    // while): latent row r by lane r / 13 of the (r % 13)-th of them, into a
    // 1040-byte pitch; the rope rows by one copy.
    const int H = p.num_heads;
    const uint32_t qbar = bar(Ctl::kQFull, 0);
    if (tid == 0) mbar_arrive_tx(qbar, static_cast<uint32_t>(H * (kLatent + kRope) * 2));
    __syncwarp();
    const uint16_t* qlat_t = p.q_lat + static_cast<int64_t>(t) * H * kLatent;
    const int qw = warp - (warp > kProducerWarp ? 1 : 0) - (warp > kCopyWarpA ? 1 : 0) -
                   (warp > kCopyWarpB ? 1 : 0);
    if (warp != kProducerWarp && !is_copy_warp(warp))
      for (int r = lane * 13 + qw; r < H && lane < 10; r += 32 * 13)
        bulk_g2s(sbase + L::kQStage + r * L::kQPitch, qlat_t + static_cast<int64_t>(r) * kLatent,
                 kLatent * 2, qbar);
    if (tid == 32)
      bulk_g2s(sbase + L::kQStage + L::kQRopeStage, p.q_rope + static_cast<int64_t>(t) * H * kRope,
               static_cast<uint32_t>(H * kRope * 2), qbar);
  }
  // Score CTA start-up: Q latent (bf16 staging rows) -> FP16 in TMEM, the QK
  // MMA's A operand, by the softmax warps (thread = head). Chunk c is 64 dims
  // (32 TMEM columns) of one head.
  auto convert_q = [&](int c0, int c1, bool live) {
    const int h = warp * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    live = live && h < p.num_heads;
#pragma unroll 1
    for (int c = c0; c < c1; ++c) {
      uint32_t r[32];
      const uint32_t src = sbase + L::kQStage + h * L::kQPitch + c * 128;
#pragma unroll
      for (int v = 0; v < 8; ++v) {
        const uint4 x = bf16x8_to_f16x8(
            live ? ld_shared_v4(src + v * 16) : make_uint4(0u, 0u, 0u, 0u), p.q_lat_mult);
        r[4 * v] = x.x;
        r[4 * v + 1] = x.y;
        r[4 * v + 2] = x.z;
        r[4 * v + 3] = x.w;
      }
      tmem_st32(tmem + lane_base + 32u * c, r);
    }
    tmem_st_wait();
  };
  const uint32_t copy = rank == 0 ? L::kCopyS : L::kCopyO;
  const uint32_t raw_base = sbase + (rank == 0 ? L::kRawS : L::kRawO);
  const uint32_t stage_bytes = rank == 0 ? L::kStageS : L::kStageO;
  const uint32_t group_bytes = rank == 0 ? L::kGroupS : L::kGroupO;
  const uint32_t row_pad = rank == 0 ? L::kRowS : L::kRowO;
  auto raw_row = [&](int s, int r) {  // row r of gather stage s
    return raw_base + s * stage_bytes + (r >> 2) * group_bytes + (r & 3) * row_pad;
  };

  const uint32_t offs_base = sbase + (rank == 0 ? L::kOffsS : L::kOffsO);
  auto offs_row = [&](int slot) { return offs_base + slot * L::kOffsSlot; };
  auto offs_mask = [&](int slot) { return offs_base + slot * L::kOffsSlot + kSub * 8; };

  // Copies of stage u, issued by the two copy warps (iw = 0, 1) as soon as
  // the stage is resolved and its ring slot released. Tensor path: lanes 0-7
  // of warp iw issue the gather4 copies of row groups 8 iw .. 8 iw + 7 (a
  // group with no live row is skipped; dead rows of a live group re-read one
  // of its live rows). Fallback (a page stride that is not a whole number of
  // rows): lane l of warp iw copies row 32 iw + l when live. A copy
  // instruction stalls its warp for a while, hence dedicated warps. One thread
  // arms the stage's barrier with the stage's byte count.
  const CUtensorMap* tmap = rank == 0 ? &tm_s : &tm_o;
  auto issue_stage = [&](int u, int iw) -> bool {
    const int os = u % L::kOffsSlots;
    const int s = u % stages;
    if (!warp_wait(bar(Ctl::kOffsFull, os), (u / L::kOffsSlots) & 1u, abort_addr)) return false;
    if (!warp_wait(bar(Ctl::kRawEmpty, s), ((u / stages) & 1u) ^ 1u, abort_addr)) return false;
    const uint64_t mask = ld_shared_u64(offs_mask(os));
    const uint32_t full = bar(Ctl::kRawFull, s);
    if (p.use_tma) {
      const uint64_t any = (mask | (mask >> 1) | (mask >> 2) | (mask >> 3)) & 0x1111111111111111ull;
      if (iw == 0 && lane == 0)
        mbar_arrive_tx(full, static_cast<uint32_t>(__popcll(any)) * 4u * row_pad);
      if (lane < 8) {
        const int g = 8 * iw + lane;
        const uint32_t m4 = static_cast<uint32_t>(mask >> (4 * g)) & 15u;
        if (m4 != 0u) {
          const int first = 4 * g + __ffs(m4) - 1;
          int32_t y[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int r = ((m4 >> k) & 1u) ? 4 * g + k : first;
            y[k] = static_cast<int32_t>(ld_shared_u64(offs_row(os) + 8 * r) / L::kRowBytes);
          }
          gather4(raw_row(s, 4 * g), tmap, y[0], y[1], y[2], y[3], full);
        }
      }
    } else {
      if (iw == 0 && lane == 0)
        mbar_arrive_tx(full, static_cast<uint32_t>(__popcll(mask)) * copy);
      const int r = 32 * iw + lane;
      if ((mask >> r) & 1ull)
        bulk_g2s(raw_row(s, r), p.cache + ld_shared_u64(offs_row(os) + 8 * r), copy, full);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(Ctl::kOffsEmpty, os));
    return true;
  };

  if (is_copy_warp(warp)) {
    // ------------------------------------------------ gather copies
    // (score CTA: Q is staged over the ring until it is converted)
    bool run = rank != 0 || warp_wait(bar(Ctl::kQReady, 0), 0, abort_addr);
    for (int u = 0; u < n_sub && run; ++u) run = issue_stage(u, warp == kCopyWarpA ? 0 : 1);
  } else if (warp == kProducerWarp) {
    // ------------------------------------------------ resolve: slots -> row offsets
    // Index and block-table loads are dependent global loads; four stages are
    // resolved per batch with all their loads in flight together, and the
    // next batch's index loads overlap this batch's block-table loads.
    const bool seq_ok = b >= 0 && b < p.num_seqs;
    const int32_t* bt_row = p.block_table + static_cast<int64_t>(seq_ok ? b : 0) * p.max_blocks;
    // page of a position: >= 0, -1 for an empty slot, -2 when it does not
    // resolve. The block-table load is issued before the length check (its
    // index is kept inside the sequence's row), so it does not wait on the
    // length load.
    auto load_page = [&](const int32_t (&pos)[2], int64_t (&pg)[2]) {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int32_t ps = pos[j];
        const int32_t pi = ps >= 0 ? ps / p.page_size : -1;
        const bool in_row = seq_ok && pi >= 0 && pi < p.max_blocks;
        const int64_t e = in_row ? __ldg(bt_row + pi) : -1;
        pg[j] = ps == -1 ? -1 : (!in_row || ps >= len || e < 0 || e >= p.num_blocks) ? -2 : e;
      }
    };
    bool stop = false;
    for (int u0 = 0; u0 < n_sub && !stop; u0 += 4) {
      int64_t pg[4][2];
      int32_t posb[4][2];
#pragma unroll
      for (int k = 0; k < 4; ++k) load_page(posa[k], pg[k]);
#pragma unroll
      for (int k = 0; k < 4; ++k) load_pos(u0 + 4 + k, posb[k]);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int u = u0 + k;
        if (u >= n_sub) break;
        const int os = u % L::kOffsSlots;
        if (!warp_wait(bar(Ctl::kOffsEmpty, os), ((u / L::kOffsSlots) & 1u) ^ 1u, abort_addr)) {
          stop = true;
          break;
        }
        bool val[2];
        int bad = 0;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          val[j] = pg[k][j] >= 0;
          bad += pg[k][j] == -2;
          const int64_t off = val[j] ? pg[k][j] * p.block_stride +
                                           static_cast<int64_t>(posa[k][j] % p.page_size) *
                                               L::kRowBytes
                                     : 0;
          st_shared_u64(offs_row(os) + 8 * (lane + 32 * j), static_cast<uint64_t>(off));
        }
        const uint32_t b0 = __ballot_sync(0xffffffffu, val[0]);
        const uint32_t b1 = __ballot_sync(0xffffffffu, val[1]);
        const uint64_t mask = (static_cast<uint64_t>(b1) << 32) | b0;
        if (rank == 0) {
          bad = __reduce_add_sync(0xffffffffu, bad);
          if (lane == 0 && bad > 0 && p.invalid_count != nullptr) atomicAdd(p.invalid_count, bad);
        }
        __syncwarp();
        if (lane == 0) {
          st_shared_u64(offs_mask(os), mask);
          *reinterpret_cast<volatile uint64_t*>(smem + L::kCtl + Ctl::kMaskRing + 8 * (u & 31)) =
              mask;
          mbar_arrive(bar(Ctl::kOffsFull, os));
        }
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        posa[k][0] = posb[k][0];
        posa[k][1] = posb[k][1];
      }
    }
  } else if (warp >= 6 && rank == 0) {
    // ------------------------------------------------ score CTA: gather + K chunks
    // Chunk kb of tile i: rows 0..127 of the tile x dims [64 kb, 64 kb + 64)
    // (kb = 8: the 64 rope dims). Thread -> (row, half of the chunk's dims).
    const int dt = dequant_index(warp) * 32 + lane;
    const int row = dt & 127;
    const int hf = dt >> 7;
    bool run = warp_wait(bar(Ctl::kQReady, 0), 0, abort_addr);  // Q staging overlaps the ring
    for (int i = 0; i < n_tiles && run; ++i) {
      const int ua = 2 * i, ub = 2 * i + 1;
      const int sa = ua % L::kStagesS, sb = ub % L::kStagesS;
      if (!warp_wait(bar(Ctl::kRawFull, sa), (ua / L::kStagesS) & 1u, abort_addr) ||
          !warp_wait(bar(Ctl::kRawFull, sb), (ub / L::kStagesS) & 1u, abort_addr))
        break;
      const int sr = row < kSub ? sa : sb;
      const int ur = row < kSub ? ua : ub;
      const uint64_t mask = *reinterpret_cast<volatile uint64_t*>(
          smem + L::kCtl + Ctl::kMaskRing + 8 * (ur & 31));
      const bool ok = (mask >> (row & 63)) & 1ull;
      // Reads below stay within bytes [0, row bytes) of the row slot (NVFP4:
      // codes < 256, scales < 288, rope < 352; FP8: < 576), so the 16 pad bytes
      // that the per-row bulk copies leave unwritten are never read.
      const uint32_t src = raw_row(sr, row & 63);
      // one chunk: wait for its ring slot, store 32 FP16 values, signal the MMA
      auto put_chunk = [&](int kb, const uint32_t (&h)[16]) -> bool {
        const int q = i * kChunksPerTile + kb;
        const int cs = q % kChunkSlots;
        if (!warp_wait(bar(Ctl::kChunkEmpty, cs), ((q / kChunkSlots) & 1u) ^ 1u, abort_addr))
          return false;
        const uint32_t dst = sbase + cs * L::kChunk;
#pragma unroll
        for (int c = 0; c < 4; ++c)
          st_shared_v4(dst + sw128_off(row, 4 * hf + c), h[4 * c], h[4 * c + 1], h[4 * c + 2],
                       h[4 * c + 3]);
        fence_proxy_async_cta();  // generic stores -> visible to the tensor core
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(Ctl::kChunkFull, cs));
        return true;
      };
      if constexpr (L::kNv) {
        // One rolled loop over the 8 latent chunks (a single copy of the
        // body keeps the hot code small); chunk kb + 1's 16 bytes of codes
        // and 4 scale bytes are loaded while chunk kb is converted.
        const uint4 z = make_uint4(0u, 0u, 0u, 0u);
        uint4 rp[2];
#pragma unroll
        for (int x = 0; x < 2; ++x) rp[x] = ok ? ld_shared_v4(src + kRopeOff + 32 * hf + 16 * x) : z;
        uint4 pay = ok ? ld_shared_v4(src + 16 * hf) : z;
        uint32_t scw = ok ? ld_shared_u32(src + kScaleOff) : 0u;
#pragma unroll 1
        for (int kb = 0; kb < 8 && run; ++kb) {
          const int kn = kb < 7 ? kb + 1 : kb;
          const uint4 pay_n = ok ? ld_shared_v4(src + 32 * kn + 16 * hf) : z;
          const uint32_t scw_n = ok ? ld_shared_u32(src + kScaleOff + 4 * kn) : 0u;
          const uint32_t sc = (scw >> (16 * hf)) & 0xFFFFu;
          const uint32_t s0 = e4m3x2_to_f16x2(static_cast<uint16_t>((sc & 0xFFu) * 0x0101u));
          const uint32_t s1 = e4m3x2_to_f16x2(static_cast<uint16_t>((sc >> 8) * 0x0101u));
          const uint32_t w[4] = {pay.x, pay.y, pay.z, pay.w};
          uint32_t h[16];
#pragma unroll
          for (int x = 0; x < 4; ++x) {
            uint32_t f[4];
            e2m1x8_to_f16x8(w[x], f);
            const uint32_t sx = x < 2 ? s0 : s1;
#pragma unroll
            for (int y = 0; y < 4; ++y) h[4 * x + y] = hmul2_u32(f[y], sx);
          }
          run = put_chunk(kb, h);
          pay = pay_n;
          scw = scw_n;
        }
        if (run) {
          uint32_t h[16], lo[8], hi[8];
          e4m3x16_to_f16(rp[0], lo);
          e4m3x16_to_f16(rp[1], hi);
#pragma unroll
          for (int x = 0; x < 8; ++x) {
            h[x] = lo[x];
            h[8 + x] = hi[x];
          }
          run = put_chunk(8, h);
        }
      } else {
#pragma unroll 1
        for (int kb = 0; kb < kChunksPerTile && run; ++kb) {
          uint32_t h[16], lo[8], hi[8];
          const uint4 z = make_uint4(0u, 0u, 0u, 0u);
          e4m3x16_to_f16(ok ? ld_shared_v4(src + 64 * kb + 32 * hf) : z, lo);
          e4m3x16_to_f16(ok ? ld_shared_v4(src + 64 * kb + 32 * hf + 16) : z, hi);
#pragma unroll
          for (int x = 0; x < 8; ++x) {
            h[x] = lo[x];
            h[8 + x] = hi[x];
          }
          run = put_chunk(kb, h);
        }
      }
      if (!run) break;
      __syncwarp();
      if (lane == 0) {  // stages sa and sb have been read: the copy warps may refill them
        mbar_arrive(bar(Ctl::kRawEmpty, sa));
        mbar_arrive(bar(Ctl::kRawEmpty, sb));
      }
    }
  } else if (warp >= 6) {
    // ------------------------------------------------ output CTA: gather + V slots
    // V (rows x 512 dims, FP16) is read by the P V MMA MN-major: each 32-row
    // slot holds 8 blocks of 64 dims, each block 4 groups of 8 rows x 128 B.
    // Thread item = (row, 16-dim group); 4 items per thread per slot.
    const int dt = dequant_index(warp) * 32 + lane;
    bool run = true;
    for (int u = 0; u < n_sub && run; ++u) {
      const int s = u % L::kStagesO;
      if (!warp_wait(bar(Ctl::kRawFull, s), (u / L::kStagesO) & 1u, abort_addr)) break;
      const uint64_t mask =
          *reinterpret_cast<volatile uint64_t*>(smem + L::kCtl + Ctl::kMaskRing + 8 * (u & 31));
#pragma unroll 1
      for (int hh = 0; hh < 2; ++hh) {
        const int hs = 2 * u + hh;
        const int vs = hs % L::kVSlots;
        if (!warp_wait(bar(Ctl::kVtEmpty, vs), ((hs / L::kVSlots) & 1u) ^ 1u, abort_addr)) {
          run = false;
          break;
        }
        const uint32_t vslot = sbase + vs * L::kVSlot;
#pragma unroll
        for (int it = 0; it < 4; ++it) {
          const int item = dt + 256 * it;
          const int r = item & 31;          // row within the slot
          const int j = item >> 5;          // 16-dim group 0..31
          const int rr = 32 * hh + r;       // row within the stage
          const uint32_t rp = raw_row(s, rr);
          const bool ok = (mask >> rr) & 1ull;
          uint32_t h[8];
          if (!ok) {
#pragma unroll
            for (int x = 0; x < 8; ++x) h[x] = 0u;
          } else if constexpr (L::kNv) {
            const uint2 pl = ld_shared_v2(rp + 8 * j);
            const uint32_t sc = ld_shared_u8(rp + kScaleOff + j);
            const uint32_t s2h = e4m3x2_to_f16x2(static_cast<uint16_t>(sc * 0x0101u));
            uint32_t lo[4], hi[4];
            e2m1x8_to_f16x8(pl.x, lo);
            e2m1x8_to_f16x8(pl.y, hi);
#pragma unroll
            for (int y = 0; y < 4; ++y) {
              h[y] = hmul2_u32(lo[y], s2h);
              h[4 + y] = hmul2_u32(hi[y], s2h);
            }
          } else {
            e4m3x16_to_f16(ld_shared_v4(rp + 16 * j), h);
          }
          // dims [16 j, 16 j + 16): block nb = j / 4, 16-byte chunks 2 (j % 4), +1
          const uint32_t blk = vslot + (j >> 2) * 4096u;
          const uint32_t c0 = static_cast<uint32_t>((j & 3) * 2);
          st_shared_v4(blk + sw128_off(r, c0), h[0], h[1], h[2], h[3]);
          st_shared_v4(blk + sw128_off(r, c0 + 1), h[4], h[5], h[6], h[7]);
        }
        fence_proxy_async_cta();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(Ctl::kVtFull, vs));
      }
      if (!run) break;
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(Ctl::kRawEmpty, s));  // stage s read: the copy warps refill it
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------ MMA issue (one thread)
    if (lane == 0) {
      uint32_t last_bar = 0, last_parity = 0;
      bool issued = false;
      if (rank == 0) {
        if (wait_bar(bar(Ctl::kQReady, 0), 0, abort_addr)) {
          // Operands from loop-invariant bases: the allocation of all 512
          // columns starts at TMEM address 0 (checked at set-up), the chunk
          // ring at the start of shared memory; a descriptor's address field
          // counts 16 bytes.
          const uint64_t qrope = sw128_desc(sbase + L::kQRope);
          const uint64_t ring = sw128_desc(sbase);
          bool run = true;
          for (int i = 0; i < n_tiles && run; ++i) {
            const int s2 = i & 1;
            const uint32_t k2 = i >> 1;
            if (!wait_bar(bar(Ctl::kSEmpty, s2), (k2 & 1u) ^ 1u, abort_addr)) break;
            const uint32_t dcol = kSCol + 128u * s2;
            for (int kb = 0; kb < kChunksPerTile; ++kb) {
              const int q = i * kChunksPerTile + kb;
              const int cs = q % kChunkSlots;
              if (!wait_bar(bar(Ctl::kChunkFull, cs), (q / kChunkSlots) & 1u, abort_addr)) {
                run = false;
                break;
              }
              tc_fence_after();
              const uint64_t bd = ring + static_cast<uint64_t>(cs * (L::kChunk >> 4));
              if (kb < 8) {
                const uint32_t a = 32u * kb;
                mma_ts(dcol, a, bd, kIdescQK, kb != 0);
                mma_ts(dcol, a + 8u, bd + 2u, kIdescQK, 1u);
                mma_ts(dcol, a + 16u, bd + 4u, kIdescQK, 1u);
                mma_ts(dcol, a + 24u, bd + 6u, kIdescQK, 1u);
              } else {
                mma_ss(dcol, qrope, bd, kIdescQK, 1u);
                mma_ss(dcol, qrope + 2u, bd + 2u, kIdescQK, 1u);
                mma_ss(dcol, qrope + 4u, bd + 4u, kIdescQK, 1u);
                mma_ss(dcol, qrope + 6u, bd + 6u, kIdescQK, 1u);
              }
              mma_commit(bar(Ctl::kChunkEmpty, cs));
              last_bar = bar(Ctl::kChunkEmpty, cs);
              last_parity = (q / kChunkSlots) & 1u;
              issued = true;
            }
            if (run) mma_commit(bar(Ctl::kSFull, s2));
          }
        }
      } else {
        uint32_t n_corr = 0;
        for (int u = 0; u < n_sub; ++u) {
          const int s2 = u & 1;
          const uint32_t k2 = u >> 1;
          // P (and any rescale of O) first; then each 32-row V slot is
          // multiplied as soon as it is full and released by its own commit,
          // so the dequant warps can refill it while the other slot's MMAs run
          if (!wait_bar<true>(bar(Ctl::kPFull, s2), k2 & 1u, abort_addr)) break;
          const uint4 fl = ld_shared_v4(ctl + Ctl::kAF + s2 * kAFBytes + 512);
          if ((fl.x | fl.y | fl.z | fl.w) != 0u) {
            if (!wait_bar(bar(Ctl::kOCorr, 0), n_corr & 1u, abort_addr)) break;
            ++n_corr;
          }
          const uint32_t ptile = sbase + L::kP + s2 * L::kPTile;
          bool run = true;
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int hs = 2 * u + hh;
            const int vs = hs % L::kVSlots;
            if (!wait_bar(bar(Ctl::kVtFull, vs), (hs / L::kVSlots) & 1u, abort_addr)) {
              run = false;
              break;
            }
            tc_fence_after();
#pragma unroll
            for (int k1 = 0; k1 < 2; ++k1) {
              const int kk = 2 * hh + k1;
              const uint64_t adesc = sw128_desc(ptile + kk * 32u);
              const uint32_t vslot = sbase + vs * L::kVSlot + k1 * 2048u;
#pragma unroll
              for (int nh = 0; nh < 2; ++nh) {
                const uint64_t bdesc = sw128_desc_mn(vslot + nh * 16384u);
                mma_ss(tmem + 256u * nh, adesc, bdesc, kIdescPV, (u > 0 || kk > 0) ? 1u : 0u);
              }
            }
            mma_commit(bar(Ctl::kVtEmpty, vs));
            last_bar = bar(Ctl::kVtEmpty, vs);  // tracks every MMA issued so far
            last_parity = (hs / L::kVSlots) & 1u;
            issued = true;
          }
          if (!run) break;
          mma_commit(bar(Ctl::kPvDone, s2));
          last_bar = bar(Ctl::kPvDone, s2);
          last_parity = k2 & 1u;
          issued = true;
        }
      }
      if (issued) drain_bar(last_bar, last_parity);  // every issued MMA has completed
    }
  } else if (rank == 0) {
    // ------------------------------------------------ score CTA: Q setup, then softmax
    const int h = warp * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    bool ok;
    {
      // Q (bf16) of this token arrives by the copies issued at set-up over the
      // still unused buffers; each thread converts its head's row to FP16
      // (scales folded in): the latent part into TMEM, the rope part into the
      // swizzled shared-memory operand.
      const uint32_t qbar = bar(Ctl::kQFull, 0);
      const uint32_t rope_at = sbase + L::kQStage + L::kQRopeStage;
      ok = group_and(wait_bar(qbar, 0, abort_addr));  // copies issued at set-up
      const bool live = ok && h < p.num_heads;
      convert_q(0, 8, ok);
      uint4 qr[8];
#pragma unroll
      for (int v = 0; v < 8; ++v)
        qr[v] = bf16x8_to_f16x8(live ? ld_shared_v4(rope_at + h * (kRope * 2) + v * 16)
                                     : make_uint4(0u, 0u, 0u, 0u),
                                p.q_rope_mult);
      __syncwarp();
      group_sync();  // every staged row has been read: the rope operand may overwrite it
#pragma unroll
      for (int v = 0; v < 8; ++v)
        st_shared_v4(sbase + L::kQRope + sw128_off(h, v), qr[v].x, qr[v].y, qr[v].z, qr[v].w);
      fence_proxy_async_cta();
      tc_fence_before();
      mbar_arrive(bar(Ctl::kQReady, 0));
    }
    const uint32_t peer_p = map_rank(sbase + L::kP, peer);
    const uint32_t peer_ctl = map_rank(ctl, peer);
    const float c = p.score_scale;
    float m_ref = -INFINITY, l = 0.f;
    for (int i = 0; i < n_tiles && ok; ++i) {
      const int s2 = i & 1;
      const uint32_t k2 = i >> 1;
      ok = group_and(ok && wait_bar(bar(Ctl::kSFull, s2), k2 & 1u, abort_addr));
      if (!ok) break;
      tc_fence_after();
      uint64_t masks[2];
      masks[0] = *reinterpret_cast<volatile uint64_t*>(smem + L::kCtl + Ctl::kMaskRing +
                                                        8 * ((2 * i) & 31));
      masks[1] = *reinterpret_cast<volatile uint64_t*>(smem + L::kCtl + Ctl::kMaskRing +
                                                        8 * ((2 * i + 1) & 31));
#pragma unroll 1
      for (int jj = 0; jj < 2; ++jj) {
        const int u = 2 * i + jj;
        const uint64_t mask = masks[jj];
        uint32_t sa[32], sb[32];
        tmem_ld32(tmem + lane_base + kSCol + 128u * s2 + 64u * jj, sa);
        tmem_ld32(tmem + lane_base + kSCol + 128u * s2 + 64u * jj + 32u, sb);
        tmem_ld_wait();
        if (jj == 1) {
          tc_fence_before();
          mbar_arrive(bar(Ctl::kSEmpty, s2));
        }
        // raw max over the valid rows (the scale c > 0 is applied once after)
        float mx = -INFINITY;
        if (mask == ~0ull) {
          float ma = -INFINITY, mb = -INFINITY;
#pragma unroll
          for (int q = 0; q < 32; q += 2) {
            ma = fmax3(ma, __uint_as_float(sa[q]), __uint_as_float(sb[q]));
            mb = fmax3(mb, __uint_as_float(sa[q + 1]), __uint_as_float(sb[q + 1]));
          }
          mx = fmaxf(ma, mb);
        } else {
#pragma unroll
          for (int q = 0; q < 32; ++q) {
            const float v0 = ((mask >> q) & 1ull) ? __uint_as_float(sa[q]) : -INFINITY;
            const float v1 = ((mask >> (32 + q)) & 1ull) ? __uint_as_float(sb[q]) : -INFINITY;
            sa[q] = __float_as_uint(v0);
            sb[q] = __float_as_uint(v1);
            mx = fmaxf(mx, fmaxf(v0, v1));
          }
        }
        const float mxs = mx * c;
        float alpha = 1.f;
        bool resc = false;
        if (mxs > m_ref + kTau) {  // also the first valid score (m_ref = -inf)
          alpha = m_ref == -INFINITY ? 0.f : ex2(m_ref - mxs);
          m_ref = mxs;
          l *= alpha;
          resc = true;
        }
        const float neg_m = m_ref == -INFINITY ? 0.f : -m_ref;
        const bool none = m_ref == -INFINITY;
        // stage P + rescale factor + flags; slot u & 1 of the staging area
        const int st = u & 1;
        const uint32_t stage = sbase + L::kPStage + st * L::kPStageStride;
        if (tid == 0) bulk_wait_read<1>();  // the copy that last used this slot has read it
        ok = group_and(ok);                 // (also carries thread 0's last send status)
        if (!ok) break;
        // P = 2^(s c - m_ref) in two halves of 32 rows; masked rows hold -inf
        // (fma gives -inf, ex2 gives 0). Pairs go through the packed fp32 ops.
        const uint64_t c2 = f32x2(c, c), nm2 = f32x2(neg_m, neg_m);
        uint64_t sum2 = f32x2(0.f, 0.f);
        auto p_half = [&](const uint32_t (&x)[32], int hx) {
          uint32_t pk[16];
#pragma unroll
          for (int q = 0; q < 16; ++q) {
            float t0, t1;
            f32x2_split(fma_f32x2(f32x2(__uint_as_float(x[2 * q]), __uint_as_float(x[2 * q + 1])),
                                  c2, nm2),
                        t0, t1);
            const float p0 = none ? 0.f : ex2(t0);
            const float p1 = none ? 0.f : ex2(t1);
            pk[q] = pack_f16x2(p0, p1);
            sum2 = add_f32x2(sum2, f32x2(p0, p1));
          }
#pragma unroll
          for (int cc = 0; cc < 4; ++cc)
            st_shared_v4(stage + sw128_off(h, 4 * hx + cc), pk[4 * cc], pk[4 * cc + 1],
                         pk[4 * cc + 2], pk[4 * cc + 3]);
        };
        p_half(sa, 0);
        p_half(sb, 1);
        float sum_lo, sum_hi;
        f32x2_split(sum2, sum_lo, sum_hi);
        l += sum_lo + sum_hi;
        st_shared_u32(stage + 16384 + 4 * h, __float_as_uint(alpha));
        const bool warp_resc = __any_sync(0xffffffffu, resc && u > 0);
        if (lane == 0) st_shared_u32(stage + 16384 + 512 + 4 * warp, warp_resc ? 1u : 0u);
        fence_proxy_async_cta();  // generic stores -> visible to the bulk copy
        group_sync();             // every thread's part of P is staged
        // Thread 0 alone waits for the peer's buffer and sends; the others go
        // on with the next sub-tile and meet it at that sub-tile's staging.
        if (tid == 0) {
          // the peer's P buffer st is free once its P V of sub-tile u-2 completed
          ok = wait_bar<true>(bar(Ctl::kPEmpty, st), ((u >> 1) & 1u) ^ 1u, abort_addr);
          if (ok) {
            const uint32_t pbar = peer_ctl + Ctl::kPFull + 8 * st;
            mbar_arrive_tx_cluster(pbar, 16384 + kAFBytes);
            bulk_s2s(peer_p + st * L::kPTile, stage, 16384, pbar);
            bulk_s2s(peer_ctl + Ctl::kAF + st * kAFBytes, stage + 16384, kAFBytes, pbar);
            bulk_commit();
          }
        }
      }
    }
    if (tid == 0) bulk_wait_read<0>();  // this CTA's staging is read before it exits
    ok = group_and(ok);
    if (ok) {
      st_cluster_u32(peer_ctl + Ctl::kFinalM + 4 * h, __float_as_uint(m_ref));
      st_cluster_u32(peer_ctl + Ctl::kFinalL + 4 * h, __float_as_uint(l));
      mbar_arrive_cluster(peer_ctl + Ctl::kStats);
    }
  } else {
    // ------------------------------------------------ output CTA: corrections + epilogue
    const int h = warp * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t peer_ctl = map_rank(ctl, peer);
    bool ok = true;
    for (int u = 0; u < n_sub; ++u) {
      const int s2 = u & 1;
      const uint32_t k2 = u >> 1;
      if (!warp_wait(bar(Ctl::kPvDone, s2), k2 & 1u, abort_addr)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // this warp has read buffer s2's flags and factors (for sub-tile u, in
      // the previous iteration): the score CTA may refill it. The reads have
      // completed (their values decided this warp's work), so a relaxed
      // arrive suffices.
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster_relaxed(peer_ctl + Ctl::kPEmpty + 8 * s2);
      if (u + 1 < n_sub) {
        const int n2 = (u + 1) & 1;
        const uint32_t nk2 = (u + 1) >> 1;
        if (!warp_wait<true>(bar(Ctl::kPFull, n2), nk2 & 1u, abort_addr)) {
          ok = false;
          break;
        }
        const uint32_t af = ctl + Ctl::kAF + n2 * kAFBytes;
        const uint4 fl = ld_shared_v4(af + 512);
        if ((fl.x | fl.y | fl.z | fl.w) != 0u) {
          const float alpha = __uint_as_float(ld_shared_u32(af + 4 * h));
#pragma unroll 1
          for (int cc = 0; cc < 16; ++cc) {
            uint32_t r[32];
            tmem_ld32(tmem + lane_base + 32u * cc, r);
            tmem_ld_wait();
#pragma unroll
            for (int q = 0; q < 32; ++q) r[q] = __float_as_uint(__uint_as_float(r[q]) * alpha);
            tmem_st32(tmem + lane_base + 32u * cc, r);
          }
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(bar(Ctl::kOCorr, 0));
        }
      }
    }
    float m_fin = NAN, l_fin = 0.f;
    ok = __all_sync(0xffffffffu, ok);
    if (ok && warp_wait<true>(bar(Ctl::kStats, 0), 0, abort_addr)) {
      m_fin = __uint_as_float(ld_shared_u32(ctl + Ctl::kFinalM + 4 * h));
      l_fin = __uint_as_float(ld_shared_u32(ctl + Ctl::kFinalL + 4 * h));
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
      // Rows leave through shared memory (V slots and P tiles are idle now):
      // each thread stages its head's row at a padded pitch (conflict-free),
      // then each warp writes its 32 rows with stores that are contiguous
      // across the warp. fp32 rows (fp32 output, split-K partials) go in two
      // halves of 256 columns so the staging stays within 133 KB.
      const bool f32 = !(single && !p.out_fp32);
      constexpr uint32_t kOutPitch = 1024 + 16;
      const uint32_t stg = sbase + static_cast<uint32_t>(h) * kOutPitch;
      const int H = p.num_heads;
#pragma unroll 1
      for (int hv = 0; hv < (f32 ? 2 : 1); ++hv) {
#pragma unroll 1
        for (int cc = 0; cc < (f32 ? 8 : 16); ++cc) {
          uint32_t r[32];
          if (ok) {
            tmem_ld32(tmem + lane_base + 256u * hv + 32u * cc, r);
            tmem_ld_wait();
          } else {
#pragma unroll
            for (int q = 0; q < 32; ++q) r[q] = 0u;
          }
          float v[32];
#pragma unroll
          for (int q = 0; q < 32; ++q) v[q] = __uint_as_float(r[q]) * sc;
          if (!f32) {
#pragma unroll
            for (int q = 0; q < 4; ++q)
              st_shared_v4(stg + cc * 64 + q * 16, pack_bf16x2(v[8 * q], v[8 * q + 1]),
                           pack_bf16x2(v[8 * q + 2], v[8 * q + 3]),
                           pack_bf16x2(v[8 * q + 4], v[8 * q + 5]),
                           pack_bf16x2(v[8 * q + 6], v[8 * q + 7]));
          } else {
#pragma unroll
            for (int q = 0; q < 8; ++q)
              st_shared_v4(stg + cc * 128 + q * 16, __float_as_uint(v[4 * q]),
                           __float_as_uint(v[4 * q + 1]), __float_as_uint(v[4 * q + 2]),
                           __float_as_uint(v[4 * q + 3]));
          }
        }
        __syncwarp();
        // the warp's rows, 1 KB each (a bf16 row or an fp32 half row)
#pragma unroll 1
        for (int rr = 0; rr < 32; ++rr) {
          const int hh = warp * 32 + rr;
          if (hh >= H) break;
          const int64_t qhh = static_cast<int64_t>(t) * H + hh;
          const int64_t phh = (static_cast<int64_t>(t) * p.num_splits + split) * H + hh;
          uint8_t* dst = !f32 ? reinterpret_cast<uint8_t*>(static_cast<uint16_t*>(p.out) + qhh * kLatent)
                         : single ? reinterpret_cast<uint8_t*>(static_cast<float*>(p.out) + qhh * kLatent + 256 * hv)
                                  : reinterpret_cast<uint8_t*>(p.ws + phh * kLatent + 256 * hv);
          const uint32_t src = sbase + static_cast<uint32_t>(hh) * kOutPitch;
#pragma unroll
          for (int k = 0; k < 2; ++k)
            *reinterpret_cast<uint4*>(dst + k * 512 + lane * 16) = ld_shared_v4(src + k * 512 + lane * 16);
        }
        __syncwarp();  // the next half overwrites this warp's staging rows
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

// cuTensorMapEncodeTiled, looked up once through the runtime
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

// The pool seen as a 2-D tensor of rows (row stride = row bytes), valid when
// the page stride is a whole number of rows; one map per gathered row width.
// The last pool seen by a host thread is cached with its maps.
struct RowMaps {
  const void* cache = nullptr;
  int64_t rows = 0;
  int fmt = -1;
  bool ok = false;
  CUtensorMap s, o;
};
thread_local RowMaps t_row_maps;

template <int kFmt>
bool row_maps(const DecodeParams& p, CUtensorMap* ms, CUtensorMap* mo) {
  using L = TcLayout<kFmt>;
  if (p.block_stride % L::kRowBytes != 0) return false;
  const int64_t rows = p.num_blocks * (p.block_stride / L::kRowBytes);
  if (rows <= 0 || rows > 0x7FFFFFFFll) return false;
  RowMaps& c = t_row_maps;
  if (!(c.cache == p.cache && c.rows == rows && c.fmt == kFmt)) {
    c.cache = p.cache;
    c.rows = rows;
    c.fmt = kFmt;
    c.ok = false;
    EncodeTiledFn enc = encode_tiled();
    if (enc != nullptr) {
      const CUtensorMapDataType dt = L::kElem == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16
                                                   : CU_TENSOR_MAP_DATA_TYPE_UINT32;
      const cuuint64_t dims[2] = {static_cast<cuuint64_t>(L::kRowElems),
                                  static_cast<cuuint64_t>(rows)};
      const cuuint64_t strides[1] = {static_cast<cuuint64_t>(L::kRowBytes)};
      const cuuint32_t es[2] = {1, 1};
      // score rows: whole row + 16 bytes past its end (out of range: zero-filled)
      const cuuint32_t box_s[2] = {static_cast<cuuint32_t>(L::kRowS / L::kElem), 1};
      // output rows: the latent part + 16 bytes of the rope (in range)
      const cuuint32_t box_o[2] = {static_cast<cuuint32_t>(L::kRowO / L::kElem), 1};
      void* base = const_cast<uint8_t*>(p.cache);
      c.ok = enc(&c.s, dt, 2, base, dims, strides, box_s, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                 CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS &&
             enc(&c.o, dt, 2, base, dims, strides, box_o, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                 CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    }
  }
  if (!c.ok) return false;
  *ms = c.s;
  *mo = c.o;
  return true;
}

template <int kFmt>
int32_t launch_fmt(const DecodeParams& p, cudaStream_t stream) {
  constexpr int smem = TcLayout<kFmt>::kBytes;
  cudaFuncSetAttribute(decode_tc_kernel<kFmt>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  const int64_t ctas = 2ll * p.num_q * p.num_splits;
  if (ctas > 0x7FFFFFFF) return NVFP4_MLA_ERR_SHAPE;
  DecodeParams q = p;
  CUtensorMap ms, mo;
  memset(&ms, 0, sizeof(ms));
  memset(&mo, 0, sizeof(mo));
  q.use_tma = row_maps<kFmt>(p, &ms, &mo) ? 1 : 0;
  decode_tc_kernel<kFmt><<<static_cast<unsigned>(ctas), kThreads, smem, stream>>>(q, ms, mo);
  return launch_status();
}

}  // namespace

int32_t launch_decode_tc(const DecodeParams& p, int row_format, cudaStream_t stream) {
  if (row_format == NVFP4_MLA_ROW_FP8_576) return launch_fmt<NVFP4_MLA_ROW_FP8_576>(p, stream);
  return launch_fmt<NVFP4_MLA_ROW_NVFP4_352>(p, stream);
}

}  // namespace nvfp4_mla
