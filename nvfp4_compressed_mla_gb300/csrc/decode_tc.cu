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
// With 128 heads, one query token's resident state does not fit one SM (the
// 128 x 512 FP32 output alone fills a whole SM's tensor memory), so each
// (token, split) unit is a 2-CTA cluster that gives each of the two
// contractions of the absorbed-MLA step its own SM:
//
//   rank 0, "score" CTA: S^T = K Q^T per 128-row tile (M = 128 rows,
//     N = the heads rounded up to 32, K = 576). The dequant warps expand the gathered rows
//     (thread = row) straight into tensor memory, where they are the MMA's A
//     operand: a ring of 128-dimension chunks, so the FP16 K tile never
//     touches shared memory. Q (FP16, all 576 dimensions of the 128 heads)
//     stays resident in shared memory as the B operand; it arrives by nine
//     2-D tensor copies and is converted in place. Four softmax warps
//     (thread = row) turn their 32 rows of S^T into P^T pieces (FP16, rows x
//     heads) against a lazy reference maximum per head, and each copies its
//     piece into the peer's memory.
//   rank 1, "output" CTA: O (128 heads x 512 FP32) lives in tensor memory.
//     Per 32-row piece: O += P V (M = 128 heads, N = 2 x 256, K = 32), P^T
//     from the peer read MN-major, V dequantised from its own gather into
//     MN-major slots. Four correction warps (thread = head) add each piece's
//     column into the softmax denominator l (the same FP16 values the MMA
//     uses), rescale O and l when the score CTA raised its reference maximum,
//     hand P buffers back, and write the normalised output at the end.
//
// Both CTAs gather their own copy of the rows: two gather warps take
// alternate 32-slot stages, resolve the stage's top-k slots through the block
// table (-1 and unresolvable slots issue no load; the index loads run four
// of the warp's stages ahead, the block-table loads two), publish the stage's live-row
// mask and copy the live rows with tile::gather4 tensor copies (four rows per
// copy; one bulk copy per row when the page stride is not a whole number of
// rows). Every wait is bounded; a
// wait that runs out sets an abort flag, the roles unwind, copies and MMAs in
// flight are drained, tensor memory is freed, and the unit's outputs are NaN.
#include <cuda.h>
#include <math.h>
#include <string.h>

#include <mutex>

#include "decode_common.cuh"

namespace nvfp4_mla {
namespace {

constexpr int kSub = 32;                     // rows per gather stage / P piece / V slot
constexpr int kPiecesPerTile = kTile / kSub;  // 4
constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr int kMmaWarp = 5, kGatherWarp = 6;  // gather warps 6 and 7
constexpr int kQWarp = 4;                     // score CTA: helps convert Q
// Score CTA: Q is converted by the softmax warps 0-3, warp 4 and the dequant
// warps 8-15 (idle until their first rows land).
constexpr int kQConverters = 13;
constexpr int kDequantWarp0 = 8;             // warps 8..15; warp w runs on sub-partition w % 4
constexpr uint32_t kTmemCols = 512;
constexpr int kQTiles = 9;                   // Q: 8 latent 64-dim tiles + the rope tile
// K ring chunks per 128-row tile: 4 latent chunks of 128 dims (64 TMEM
// columns, 8 MMAs each) and the rope (64 dims, 4 MMAs). Large chunks keep the
// single MMA-issuing thread's per-chunk handshake (barrier test, fence,
// commit) off the tensor pipe's critical path.
constexpr int kChunksPerTile = 5;
constexpr int kPBufs = 6;                    // output CTA: P pieces in flight
// Gather stage u lands in data slot u % stages but completes and is released
// on barrier pair u % 8. The score CTA's four quadrant warps wait for four
// consecutive stages at once; with fewer than four data slots, a barrier per
// data slot would let a waiter be two phases ahead of it (and a parity wait
// cannot tell those phases apart). With at least four pairs, and no fewer
// than the data slots, every waiter is at most one phase ahead.
constexpr int kRawBars = 8;
// Lazy rescale threshold (log2 units): a head's reference maximum moves only
// when a score exceeds it by more than kTau, so P = 2^(s c - m_ref) <= 2^15,
// which FP16 holds (largest finite value 65504); l <= 2^15 x top-k stays far
// inside FP32. A P value is never below its exact-maximum counterpart, so the
// headroom costs no precision.
constexpr float kTau = 15.0f;
constexpr long long kDrainCycles = 1ll << 31;
// tcgen05 instruction descriptors (kind::f16, FP16 A/B, FP32 D):
//   bit 4 D = f32, bit 15 A MN-major, bit 16 B MN-major, N >> 3 at 17, M >> 4 at 24
// QK: N = the live heads rounded up to 32 (the softmax reads 32-column head chunks)
__host__ __device__ constexpr int qk_n(int num_heads) {
  return num_heads >= 128 ? 128 : (num_heads + 31) / 32 * 32;
}
// Q rows copied per tile: the live heads rounded up to 8 (rows past them are zeroed)
__host__ __device__ constexpr int q_rows(int num_heads) {
  return num_heads >= 128 ? 128 : (num_heads + 7) / 8 * 8;
}
__device__ __forceinline__ uint32_t idesc_qk(int num_heads) {
  return (1u << 4) | ((static_cast<uint32_t>(qk_n(num_heads)) >> 3) << 17) | ((128u >> 4) << 24);
}
constexpr uint32_t kIdescPV =
    (1u << 4) | (1u << 15) | (1u << 16) | ((256u >> 3) << 17) | ((128u >> 4) << 24);
constexpr uint32_t kAFBytes = 528;           // rescale factors of 128 heads + 4 flag words
constexpr uint32_t kFlagBytes = 16;          // the flag words alone (pieces 1-3 of a tile)
constexpr uint32_t kPiece = 8192;            // P^T piece: 32 rows x 128 heads FP16 (MN-major)

template <int kFmt>
struct TcLayout {
  static constexpr bool kNv = kFmt == NVFP4_MLA_ROW_NVFP4_352;
  static constexpr int kRowBytes = kNv ? kNvfp4Row : kFp8Row;
  static constexpr int kElem = kNv ? 2 : 4;                 // tensor-map element bytes
  static constexpr int kRowElems = kRowBytes / kElem;       // 176 / 144
  // Tensor memory of the score CTA: K ring (4 slots of 64 columns, one
  // 128-dimension chunk each), then two S^T buffers (128 columns each).
  static constexpr int kKSlots = 4;
  static constexpr int kSBufs = 2;
  static constexpr uint32_t kSCol = 256u;
  static_assert(64u * kKSlots <= kSCol && kSCol + 128u * kSBufs <= kTmemCols,
                "tensor memory plan");
  // Gathered rows, four per tensor copy; groups start 128-byte aligned.
  // Score CTA: whole rows. Output CTA: the latent part (NVFP4: codes and
  // scales, 288 bytes; FP8: the 512 latent bytes plus 16 of the rope, so the
  // row pitch is an odd number of 16-byte units).
  static constexpr int kRowS = kRowBytes;                   // 352 / 576
  static constexpr int kRowO = kNv ? 288 : 528;
  static constexpr int kCopyO = kNv ? 288 : 512;            // per-row bulk copies (fallback)
  static constexpr int kGroupS = (4 * kRowS + 127) / 128 * 128;  // 1408 / 2304
  static constexpr int kGroupO = (4 * kRowO + 127) / 128 * 128;  // 1152 / 2176
  static constexpr int kStageS = (kSub / 4) * kGroupS;
  static constexpr int kStageO = (kSub / 4) * kGroupO;
  // P^T pieces reach the output CTA either through a local staging slot and
  // one bulk copy per piece (NVFP4 rows), or as the softmax warps' own stores
  // into the peer (FP8 rows: the staging's 32 KB buy the score CTA's ring
  // stages of the wider rows instead; the stores are slower, the deeper
  // gather prefetch wins for those rows). The score CTA's ring holds four
  // stages (one tile) in both formats; the output CTA's three FP8 stages
  // measure as fast as four.
  static constexpr bool kDirectP = !kNv;
  static constexpr int kStagesS = 4;
  static constexpr int kStagesO = kNv ? 4 : 3;
  // score CTA
  static constexpr int kQTile = 16384;                      // 128 heads x 64 dims (SW128)
  static constexpr int kQ = 0;                              // 9 tiles: 8 latent + rope
  static constexpr int kRawS = kQ + kQTiles * kQTile;
  static constexpr int kStg = kRawS + kStagesS * kStageS;   // 4 P^T staging slots (NVFP4)
  static constexpr int kNegM = kStg + (kDirectP ? 0 : kPiecesPerTile * kPiece);  // -(ref. maximum)
  static constexpr int kAlpha = kNegM + 512;                // rescale factor per head
  static constexpr int kFlags = kAlpha + 512;               // per softmax warp: "rescaled"
  static constexpr int kAFS = kFlags + 16;                  // factors + flags of slot 0, flags 1-3
  static constexpr int kColMax = kAFS + kAFBytes + 3 * kFlagBytes;  // per softmax warp: column maxima
  static constexpr int kEndS = kColMax + kPiecesPerTile * 512;
  // output CTA
  static constexpr int kVSlot = 32 * 1024;                  // 32 rows x 512 dims FP16 (MN-major)
  // A V slot is refilled once the P V MMAs of the piece kVSlots back have
  // completed and the slot has been dequantised again, so the slot count
  // sets how many pieces the output CTA keeps in flight: four where shared
  // memory allows (NVFP4), three for the wider FP8 gather stages.
  static constexpr int kVSlots = kNv ? 4 : 3;
  static constexpr int kP = kVSlots * kVSlot;               // kPBufs P^T pieces
  static constexpr int kRawO = kP + kPBufs * kPiece;
  static constexpr int kAFO = kRawO + kStagesO * kStageO;  // factors + flags per P buffer
  static constexpr int kFinO = kAFO + kPBufs * kAFBytes;    // final reference maximum per head
  static constexpr int kScO = kFinO + 512;                  // output scale per head (epilogue)
  static constexpr int kEpiOk = kScO + 512;                 // the unit's outputs are valid
  static constexpr int kEndO = kEpiOk + 16;
  static constexpr int kCtl = ((kEndS > kEndO ? kEndS : kEndO) + 15) / 16 * 16;
  static constexpr int kCtlBytes = 1056;
  static constexpr int kBytes = kCtl + kCtlBytes;
  static_assert(kBytes <= 232448, "shared memory budget");
  static_assert(kStg % 1024 == 0 && kP % 1024 == 0, "SW128 operand alignment");
  static_assert(kRawS % 128 == 0 && kRawO % 128 == 0 && kGroupS % 128 == 0 && kGroupO % 128 == 0,
                "tensor-copy destinations");
  static_assert(kAFS % 16 == 0 && kAFO % 16 == 0, "bulk-copy alignment of the factors");
  static_assert(128 * (1024 + 16) <= kRawO + kStagesO * kStageO, "epilogue staging fits");
};

// Control block (barriers and a few words): same offset in both CTAs of the cluster.
struct Ctl {
  static constexpr int kRawFull = 0, kRawEmpty = 64, kChunkFull = 192, kChunkEmpty = 264, kSFull = 336, kSEmpty = 352,
                       kSentCnt = 368, kSent = 400, kQFull = 440,
                       kQReady = 448, kVtFull = 456, kPFull = 504, kPEmpty = 552,
                       kPvDone = 600, kOCorr = 648, kStats = 656, kSentBar = 664, kTmem = 672,
                       kAbort = 676, kMaskRing = 704, kLastStage = 960,
                       kEnd = 992;
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
// Non-blocking phase test (never suspends the thread); cluster-scope acquire
// for barriers that the peer CTA arrives on.
template <bool kCluster = false>
__device__ __forceinline__ bool mbar_ready(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  if constexpr (kCluster)
    asm volatile(
        "{\n.reg .pred p;\n"
        "mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
        "selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
  else
    asm volatile(
        "{\n.reg .pred p;\n"
        "mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n"
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
__device__ __forceinline__ uint32_t ld_shared_u16(uint32_t addr) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr) : "memory");
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
__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
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
// Arrives on `bar` once every tcgen05 operation this thread issued before it has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::
                   "r"(bar)
               : "memory");
}
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
// complete_tx, so no release ordering is needed.
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
// Barrier 1 over the 128 threads of warps 0-3, returning the OR / AND of `v` over them.
__device__ __forceinline__ bool group_or(bool v) {
  uint32_t r;
  asm volatile(
      "{\n.reg .pred p, q;\nsetp.ne.u32 p, %1, 0;\n"
      "bar.red.or.pred q, 1, 128, p;\nselp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"(v ? 1u : 0u)
      : "memory");
  return r != 0;
}
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
// Barrier 2 over the output CTA's epilogue warps: 0-3 and 8-15 (384 threads).
__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 2, 384;" ::: "memory"); }

// four rows (y0..y3) of a 2-D tensor map, one box each, into consecutive boxes at dst
__device__ __forceinline__ void gather4(uint32_t dst, const CUtensorMap* tm, int32_t y0, int32_t y1,
                                        int32_t y2, int32_t y3, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(0), "r"(y0), "r"(y1), "r"(y2), "r"(y3), "r"(bar)
      : "memory");
}
// one box of a 2-D tensor map at (x, y)
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* tm, int32_t x,
                                            int32_t y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart (stride byte offset), descriptor version 1.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t addr) {
  return static_cast<uint64_t>((addr >> 4) & 0x3FFFu) | (static_cast<uint64_t>(1) << 16) |
         (static_cast<uint64_t>(1024 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
         (static_cast<uint64_t>(2) << 61);
}
// The same for an MN-major operand whose 64-element blocks along M or N are
// 4096 bytes apart (leading byte offset) and whose 8-row groups along K are
// 1024 bytes apart (stride byte offset).
__device__ __forceinline__ uint64_t sw128_desc_mn(uint32_t addr) {
  return static_cast<uint64_t>((addr >> 4) & 0x3FFFu) | (static_cast<uint64_t>(4096 >> 4) << 16) |
         (static_cast<uint64_t>(1024 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
         (static_cast<uint64_t>(2) << 61);
}
// Byte offset of 16-byte chunk `chunk` (0..7) of row `row` in a 128-byte
// swizzled tile with 128-byte rows (8-row groups of 1024 bytes).
__device__ __forceinline__ uint32_t sw128_off(uint32_t row, uint32_t chunk) {
  return (row >> 3) * 1024u + (row & 7u) * 128u + ((chunk ^ (row & 7u)) << 4);
}

// Bounded waits. try_wait with a suspend-time hint: a waiting thread sleeps
// until the phase completes (or the hint expires) instead of spinning. The
// hint is 20 us, shorter for a short wait bound (so that the bound is kept).
__device__ __forceinline__ uint32_t suspend_ns(long long limit) {
  return limit >= 40000 ? 20000u : static_cast<uint32_t>(limit / 2 + 1);
}
template <bool kCluster>
__device__ __forceinline__ bool mbar_wait_suspend(uint32_t bar, uint32_t parity, uint32_t hint) {
  uint32_t ok;
  if constexpr (kCluster)
    asm volatile(
        "{\n.reg .pred p;\n"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n"
        "selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(hint)
        : "memory");
  else
    asm volatile(
        "{\n.reg .pred p;\n"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n"
        "selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(hint)
        : "memory");
  return ok != 0;
}
// Waits for the phase of `bar` with `parity`; false when `limit` clock
// cycles pass first (the abort flag is then set) or another thread of the
// CTA has aborted.
//
// The test that finds the phase complete is inlined; the waiting loop is one
// out-of-line copy per scope. The kernel's roles run side by side from
// different parts of a large body of code, so every copy of a cold path
// inlined into a hot loop costs instruction-cache space that the loops need.
template <bool kCluster>
__device__ __noinline__ bool wait_bar_slow(uint32_t bar, uint32_t parity, uint32_t abort_addr,
                                           long long limit) {
  const long long t0 = clock64();
  const uint32_t hint = suspend_ns(limit);
  while (true) {
    if (mbar_wait_suspend<kCluster>(bar, parity, hint)) return true;
    if (ld_shared_u32(abort_addr) != 0) return false;
    if (clock64() - t0 > limit) {
      st_shared_u32(abort_addr, 1u);
      return false;
    }
  }
}
template <bool kCluster = false>
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, uint32_t abort_addr,
                                         long long limit) {
  return mbar_test<kCluster>(bar, parity) || wait_bar_slow<kCluster>(bar, parity, abort_addr, limit);
}
// The same wait with its loop inlined, for the MMA thread's critical path.
template <bool kCluster = false>
__device__ __forceinline__ bool wait_bar_hot(uint32_t bar, uint32_t parity, uint32_t abort_addr,
                                             long long limit) {
  if (mbar_test<kCluster>(bar, parity)) return true;
  const long long t0 = clock64();
  const uint32_t hint = suspend_ns(limit);
  while (true) {
    if (mbar_wait_suspend<kCluster>(bar, parity, hint)) return true;
    if (ld_shared_u32(abort_addr) != 0) return false;
    if (clock64() - t0 > limit) {
      st_shared_u32(abort_addr, 1u);
      return false;
    }
  }
}
// Warp-uniform bounded wait: every lane waits (and so acquires) and the
// warp leaves together, so warp-collective operations after it stay converged.
template <bool kCluster = false>
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, uint32_t abort_addr,
                                          long long limit) {
  return __all_sync(0xffffffffu, wait_bar<kCluster>(bar, parity, abort_addr, limit));
}
// Bounded wait that ignores the abort flag: drains copies and MMAs that were
// issued before tensor memory is freed and the CTA exits.
template <bool kCluster = false>
__device__ __forceinline__ void drain_bar(uint32_t bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_test<kCluster>(bar, parity) && clock64() - t0 < kDrainCycles) {
  }
}

// Packed fp32 pairs (sm_100 family): one instruction does two lanes' worth
// of fma; three-input max.
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
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// bf16x8 (one 16-byte chunk) -> f16x8, each value times m (exact for m = 1)
__device__ __forceinline__ uint4 bf16x8_to_f16x8(uint4 x, float m) {
  return make_uint4(pack_f16x2(bf16_lo(x.x) * m, bf16_hi(x.x) * m),
                    pack_f16x2(bf16_lo(x.y) * m, bf16_hi(x.y) * m),
                    pack_f16x2(bf16_lo(x.z) * m, bf16_hi(x.z) * m),
                    pack_f16x2(bf16_lo(x.w) * m, bf16_hi(x.w) * m));
}
// E4M3 bytes (16) -> FP16 (16 values = 8 f16x2 words at h[0..7])
__device__ __forceinline__ void e4m3x16_to_f16(uint4 v, uint32_t* h) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    h[2 * q] = e4m3x2_to_f16x2(static_cast<uint16_t>(w[q] & 0xFFFFu));
    h[2 * q + 1] = e4m3x2_to_f16x2(static_cast<uint16_t>(w[q] >> 16));
  }
}
// f16x2 with both halves equal to the E4M3 scale byte in the low 8 bits of `b` (exact)
__device__ __forceinline__ uint32_t scale_f16x2(uint32_t b) {
  return e4m3x2_to_f16x2(static_cast<uint16_t>((b & 0xFFu) * 0x0101u));
}
// 64 dims of an NVFP4 row: 8 code words (16-dim groups g = words 2g, 2g + 1)
// times the four group scales (bytes of `scw`) -> 32 f16x2 words
__device__ __forceinline__ void nvfp4_chunk(const uint32_t (&w)[8], uint32_t scw,
                                            uint32_t (&h)[32]) {
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    const uint32_t sg = scale_f16x2(scw >> (8 * g));
#pragma unroll
    for (int x = 0; x < 2; ++x) {
      uint32_t f[4];
      e2m1x8_to_f16x8(w[2 * g + x], f);
#pragma unroll
      for (int y = 0; y < 4; ++y) h[8 * g + 4 * x + y] = hmul2_u32(f[y], sg);
    }
  }
}

// Warp reduce-scatter of the maximum: lane l returns max over all lanes of v[l].
__device__ __forceinline__ float warp_colmax(float (&v)[32], int lane) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int k = 0; k < o; ++k) {
      const float send = up ? v[k] : v[k + o];
      const float keep = up ? v[k + o] : v[k];
      v[k] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, o));
    }
  }
  return v[0];
}

// Output CTA epilogue, shared by the four correction warps and the eight V
// dequant warps (idle by then): warp (quadrant q, part) reads columns chunk
// cc = part, part + 3, ... of its quadrant's 32 heads from TMEM, scales them
// by the head's factor and stages them in the head's row in shared memory
// (over the V slots and P buffers, which every reader has finished with at
// the first barrier); then warp e of 12 writes rows e, e + 12, ... with
// stores that are contiguous across the warp. fp32 rows (fp32 output,
// split-K partials) go in two halves of 256 columns. Every warp passes the
// same barriers: the first one always, then two per half when the unit's
// outputs are valid.
// One out-of-line copy serves both callers (instruction-cache space).
template <class L>
__device__ __noinline__ void epilogue_rows(uint32_t sbase, uint32_t tmem, int q, int part, int e,
                                           int t, int split, int num_heads, int num_splits,
                                           int out_fp32, void* out, float* ws) {
  const int lane = threadIdx.x & 31;
  epi_sync();  // the factors and the valid flag are published; every P / V reader is done
  if (ld_shared_u32(sbase + L::kEpiOk) == 0u) return;
  tc_fence_after();
  constexpr uint32_t kOutPitch = 1024 + 16;
  const int h = 32 * q + lane;
  const float sc = __uint_as_float(ld_shared_u32(sbase + L::kScO + 4 * h));
  const uint32_t lq = static_cast<uint32_t>(32 * q) << 16;
  const bool single = num_splits == 1;
  const bool f32 = !(single && !out_fp32);
  const int H = num_heads;
  const uint32_t stg = sbase + static_cast<uint32_t>(h) * kOutPitch;
#pragma unroll 1
  for (int hv = 0; hv < (f32 ? 2 : 1); ++hv) {
#pragma unroll 1
    for (int cc = part; cc < (f32 ? 8 : 16); cc += 3) {
      uint32_t r[32];
      tmem_ld32(tmem + lq + 256u * hv + 32u * cc, r);
      tmem_ld_wait();
      float v[32];
#pragma unroll
      for (int k = 0; k < 32; ++k) v[k] = __uint_as_float(r[k]) * sc;
      if (!f32) {
#pragma unroll
        for (int k = 0; k < 4; ++k)
          st_shared_v4(stg + cc * 64 + k * 16, pack_bf16x2(v[8 * k], v[8 * k + 1]),
                       pack_bf16x2(v[8 * k + 2], v[8 * k + 3]),
                       pack_bf16x2(v[8 * k + 4], v[8 * k + 5]),
                       pack_bf16x2(v[8 * k + 6], v[8 * k + 7]));
      } else {
#pragma unroll
        for (int k = 0; k < 8; ++k)
          st_shared_v4(stg + cc * 128 + k * 16, __float_as_uint(v[4 * k]),
                       __float_as_uint(v[4 * k + 1]), __float_as_uint(v[4 * k + 2]),
                       __float_as_uint(v[4 * k + 3]));
      }
    }
    epi_sync();  // every row staged
    // rows of 1 KB (a bf16 row or an fp32 half row)
#pragma unroll 1
    for (int hh = e; hh < H; hh += 12) {
      const int64_t qhh = static_cast<int64_t>(t) * H + hh;
      const int64_t phh = (static_cast<int64_t>(t) * num_splits + split) * H + hh;
      uint8_t* dst =
          !f32 ? reinterpret_cast<uint8_t*>(static_cast<uint16_t*>(out) + qhh * kLatent)
          : single
              ? reinterpret_cast<uint8_t*>(static_cast<float*>(out) + qhh * kLatent + 256 * hv)
              : reinterpret_cast<uint8_t*>(ws + phh * kLatent + 256 * hv);
      const uint32_t src = sbase + static_cast<uint32_t>(hh) * kOutPitch;
#pragma unroll
      for (int k = 0; k < 2; ++k)
        *reinterpret_cast<uint4*>(dst + k * 512 + lane * 16) = ld_shared_v4(src + k * 512 + lane * 16);
    }
    epi_sync();  // every row written: the next half may overwrite the staging
  }
}

// Score CTA: converter g (0..415) turns its share of Q (bf16, as loaded)
// into FP16 in place, scales folded in, heads >= H zeroed: 16-byte item i =
// g + 416 k is chunk i % 8 of head (i / 8) % 128 of tile i / 1024 (a quarter
// warp covers one 128-byte row: no bank conflicts). Then the warp signals
// QReady. A warp whose wait for the Q copies failed converts nothing. One
// out-of-line copy serves the three roles that convert.
template <class L>
__device__ __noinline__ void convert_q_share(uint32_t sbase, uint32_t ctl, int g, int num_heads,
                                             float lat_mult, float rope_mult, uint32_t abort_addr,
                                             long long lim) {
  const bool qok = warp_wait(ctl + Ctl::kQFull, 0, abort_addr, lim);
  if (qok) {
    constexpr int kItems = kQTiles * 128 * 8;
#pragma unroll 1
    for (int i = g; i < kItems; i += 32 * kQConverters) {
      const int kb = i >> 10, h = (i >> 3) & 127, c = i & 7;
      const float m = kb < 8 ? lat_mult : rope_mult;
      const uint32_t a = sbase + L::kQ + kb * L::kQTile +
                         sw128_off(static_cast<uint32_t>(h), static_cast<uint32_t>(c));
      const uint4 x = h < num_heads ? bf16x8_to_f16x8(ld_shared_v4(a), m)
                                    : make_uint4(0u, 0u, 0u, 0u);
      st_shared_v4(a, x.x, x.y, x.z, x.w);
    }
  }
  fence_proxy_async_cta();  // generic stores -> visible to the MMA's operand reads
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(ctl + Ctl::kQReady);
}

// Score CTA softmax warps (thread tid = head h), the rare path of a tile:
// column maxima of each warp's live rows of S^T (TMEM columns from `scol_addr`,
// this warp's lanes), then per head over the four warps; a head whose scaled
// maximum exceeds its reference by more than tau moves its reference there,
// with the factor alpha that rescales what was accumulated against the old
// one (0 when there was none). Per warp, a flag says whether any of its heads
// moved after the unit's first tile. Out of line: it runs on a unit's first
// tile and rarely after, and stays out of the hot loop's instruction space.
template <class L>
__device__ __noinline__ void softmax_new_refs(uint32_t sbase, uint32_t scol_addr, bool live, float c,
                                              bool not_first) {
  const int tid = threadIdx.x, lane = tid & 31, q4 = tid >> 5;
  const uint32_t colmax = sbase + L::kColMax + q4 * 512;
#pragma unroll 1
  for (int hc = 0; hc < 4; ++hc) {
    uint32_t sv[32];
    tmem_ld32(scol_addr + 32u * hc, sv);
    tmem_ld_wait();
    float v[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = live ? __uint_as_float(sv[j]) : -INFINITY;
    st_shared_u32(colmax + 4 * (32 * hc + lane), __float_as_uint(warp_colmax(v, lane)));
  }
  group_sync();
  const int h = tid;
  float mx = -INFINITY;
#pragma unroll
  for (int w = 0; w < 4; ++w)
    mx = fmaxf(mx, __uint_as_float(ld_shared_u32(sbase + L::kColMax + w * 512 + 4 * h)));
  const float mxs = mx * c;
  const float m_old = -__uint_as_float(ld_shared_u32(sbase + L::kNegM + 4 * h));
  float alpha = 1.f;
  bool resc = false;
  if (mxs > m_old + kTau) {  // also the first live score (m_old = -inf)
    alpha = m_old == -INFINITY ? 0.f : ex2(m_old - mxs);
    st_shared_u32(sbase + L::kNegM + 4 * h, __float_as_uint(-mxs));
    resc = true;
  }
  st_shared_u32(sbase + L::kAlpha + 4 * h, __float_as_uint(alpha));
  const bool wr = __any_sync(0xffffffffu, resc) && not_first;
  if (lane == 0) st_shared_u32(sbase + L::kFlags + 4 * q4, wr ? 1u : 0u);
}

// ------------------------------------------------------------------ kernel
template <int kFmt>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    decode_tc_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap tm_s,
                     const __grid_constant__ CUtensorMap tm_o,
                     const __grid_constant__ CUtensorMap tm_ql,
                     const __grid_constant__ CUtensorMap tm_qr) {
  using L = TcLayout<kFmt>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  const uint32_t ctl = sbase + L::kCtl;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_rank();
  const uint32_t peer = rank ^ 1u;
  const long long lim = p.wait_cycles;

  const int unit = static_cast<int>(blockIdx.x >> 1);
  const int split = unit % p.num_splits;
  const int t = unit / p.num_splits;
  const int tile0 = split * p.tiles_per_split;
  const int n_tiles = min(p.tiles_per_split, p.num_tiles - tile0);
  const int n_pc = kPiecesPerTile * n_tiles;  // 32-row stages / pieces of this unit

  // The gather warps' first global loads (sequence, length, the top-k slots of
  // their first four stages) go out before the set-up, so their latency overlaps it.
  const int32_t b = __ldg(p.q_seq + t);
  const int32_t len = (b >= 0 && b < p.num_seqs) ? __ldg(p.seq_lens + b) : 0;
  const int32_t* idx_row = p.topk_idx + static_cast<int64_t>(t) * p.topk;
  auto load_pos = [&](int u) -> int32_t {
    const int slot = tile0 * kTile + u * kSub + lane;
    return (u < n_pc && slot < p.topk) ? __ldg(idx_row + slot) : -1;
  };
  const int gw = warp - kGatherWarp;  // gather warp gw takes stages gw, gw + 2, gw + 4, ...
  int32_t pos0 = -1, pos1 = -1, pos2 = -1, pos3 = -1;  // top-k slots of its next four stages
  if (gw == 0 || gw == 1) {
    pos0 = load_pos(gw);
    pos1 = load_pos(gw + 2);
    pos2 = load_pos(gw + 4);
    pos3 = load_pos(gw + 6);
  }

  auto bar = [&](int off, int i) { return ctl + off + 8u * static_cast<uint32_t>(i); };
  const uint32_t abort_addr = ctl + Ctl::kAbort;
  const int stages = rank == 0 ? L::kStagesS : L::kStagesO;

  if (tid == 0) {
    for (int s = 0; s < kRawBars; ++s) {
      mbar_init(bar(Ctl::kRawFull, s), 1);  // armed with the stage's bytes, then the copies
      mbar_init(bar(Ctl::kRawEmpty, s), rank == 0 ? 2 : 8);
      st_shared_u32(ctl + Ctl::kLastStage + 4 * s, 0u);
    }
    for (int s = 0; s < L::kKSlots; ++s) {
      mbar_init(bar(Ctl::kChunkFull, s), 4);  // the four quadrant warps of one dequant set
      mbar_init(bar(Ctl::kChunkEmpty, s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(Ctl::kSFull, s), 1);
      mbar_init(bar(Ctl::kSEmpty, s), 4);
    }
    for (int s = 0; s < kPBufs; ++s) {
      st_shared_u32(ctl + Ctl::kSentCnt + 4 * s, 0u);
      st_shared_u32(ctl + Ctl::kSent + 4 * s, 0u);
    }
    for (int s = 0; s < L::kVSlots; ++s) mbar_init(bar(Ctl::kVtFull, s), 8);
    for (int s = 0; s < kPBufs; ++s) {
      // the bulk copy's arrive + bytes, or each lane of the sending warp
      mbar_init(bar(Ctl::kPFull, s), L::kDirectP ? 32 : 1);
      mbar_init(bar(Ctl::kPEmpty, s), 4);
      mbar_init(bar(Ctl::kPvDone, s), 1);
    }
    mbar_init(bar(Ctl::kQFull, 0), 1);
    mbar_init(bar(Ctl::kQReady, 0), kQConverters);
    mbar_init(bar(Ctl::kOCorr, 0), 128);
    mbar_init(bar(Ctl::kStats, 0), 128);
    mbar_init(bar(Ctl::kSentBar, 0), 1);
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

  // Score CTA: Q of this token (bf16, the rows from row t * H: the live heads
  // rounded up to 8; rows of other tokens, past the end or past the copied
  // ones are zeroed at conversion) by nine 2-D tensor copies into
  // 128-byte-swizzled tiles, the layout of the MMA's B operand.
  if (rank == 0 && tid == 32) {
    const uint32_t qbar = bar(Ctl::kQFull, 0);
    mbar_arrive_tx(qbar, static_cast<uint32_t>(kQTiles * 128 * q_rows(p.num_heads)));
    const int32_t y = t * p.num_heads;
    for (int kb = 0; kb < 8; ++kb)
      tma_load_2d(sbase + L::kQ + kb * L::kQTile, &tm_ql, 64 * kb, y, qbar);
    tma_load_2d(sbase + L::kQ + 8 * L::kQTile, &tm_qr, 0, y, qbar);
  }

  const uint32_t raw_base = sbase + (rank == 0 ? L::kRawS : L::kRawO);
  const uint32_t stage_bytes = rank == 0 ? L::kStageS : L::kStageO;
  const uint32_t group_bytes = rank == 0 ? L::kGroupS : L::kGroupO;
  const uint32_t row_pad = rank == 0 ? L::kRowS : L::kRowO;
  auto raw_row = [&](int s, int r) {  // row r (0..31) of gather stage s
    return raw_base + s * stage_bytes + (r >> 2) * group_bytes + (r & 3) * row_pad;
  };
  auto mask_of = [&](int u) {  // live-row mask of stage u (published by its gather warp)
    return *reinterpret_cast<volatile uint32_t*>(smem + L::kCtl + Ctl::kMaskRing + 8 * (u & 31));
  };
  auto epilogue = [&](int q, int part, int e) {
    epilogue_rows<L>(sbase, tmem, q, part, e, t, split, p.num_heads, p.num_splits, p.out_fp32,
                     p.out, p.ws);
  };
  auto convert_q = [&](int g) {
    convert_q_share<L>(sbase, ctl, g, p.num_heads, p.q_lat_mult, p.q_rope_mult, abort_addr, lim);
  };

  if (gw == 0 || gw == 1) {
    // ------------------------------------------------ resolve + gather (two warps, alternate stages)
    // A copy instruction is accepted only every hundred or more cycles and the
    // slot -> page -> row chain is two dependent global loads, so two warps
    // share the stages: warp 6 the even ones, warp 7 the odd ones. Lane j
    // resolves slot j of the stage; the block-table loads run two of the
    // warp's stages ahead and the index loads four. Each stage has its own
    // barrier pair, so the two warps never share one. Stage u: the live-row
    // mask goes to the mask ring, the barrier is armed with the stage's byte
    // count, and lanes 0-7 issue the gather4 copies of row groups 0-7 (a group
    // with no live row is skipped; dead rows of a live group re-read one of
    // its live rows). Fallback (a page stride that is not a whole number of
    // rows): lane j copies row j when live. The last use of each barrier pair
    // is recorded for the drain at teardown.
    const bool seq_ok = b >= 0 && b < p.num_seqs;
    const int32_t* bt_row = p.block_table + static_cast<int64_t>(seq_ok ? b : 0) * p.max_blocks;
    const bool pow2 = (p.page_size & (p.page_size - 1)) == 0;
    const int psh = __ffs(p.page_size) - 1;
    auto page_of = [&](int32_t ps) { return pow2 ? ps >> psh : ps / p.page_size; };
    auto in_page = [&](int32_t ps) { return pow2 ? ps & (p.page_size - 1) : ps % p.page_size; };
    // page of a position: >= 0, -1 for an empty slot, -2 when it does not
    // resolve. The block-table load is issued before the length check (its
    // index is kept inside the sequence's row), so it does not wait on the
    // length load.
    auto load_page = [&](int32_t ps) -> int64_t {
      const int32_t pi = ps >= 0 ? page_of(ps) : -1;
      const bool in_row = seq_ok && pi >= 0 && pi < p.max_blocks;
      const int64_t e = in_row ? __ldg(bt_row + pi) : -1;
      return ps == -1 ? -1 : (!in_row || ps >= len || e < 0 || e >= p.num_blocks) ? -2 : e;
    };
    const CUtensorMap* tmap = rank == 0 ? &tm_s : &tm_o;
    const uint32_t copy = rank == 0 ? static_cast<uint32_t>(L::kRowS)
                                    : static_cast<uint32_t>(L::kCopyO);
    const int64_t rows_per_page = p.block_stride / L::kRowBytes;  // whole rows (tensor-map path)
    int64_t pg0 = load_page(pos0), pg1 = load_page(pos1);
    for (int u = gw; u < n_pc; u += 2) {
      const int64_t pg2 = load_page(pos2);          // stage u + 4
      const int32_t pos4 = load_pos(u + 8);         // stage u + 8
      const bool val = pg0 >= 0;
      const uint32_t mask = __ballot_sync(0xffffffffu, val);
      if (rank == 0) {
        const int bad = __popc(__ballot_sync(0xffffffffu, pg0 == -2));
        if (lane == 0 && bad > 0 && p.invalid_count != nullptr) atomicAdd(p.invalid_count, bad);
      }
      const int s = u % stages;  // data slot
      if (u >= stages) {  // data slot s is free once stage u - stages was released
        const int v = u - stages;
        if (!warp_wait(bar(Ctl::kRawEmpty, v % kRawBars), (v / kRawBars) & 1u, abort_addr, lim))
          break;
      }
      const uint32_t full = bar(Ctl::kRawFull, u % kRawBars);
      // the mask is stored before the arrive (release) that the dequant warps acquire
      if (lane == 0)
        *reinterpret_cast<volatile uint64_t*>(smem + L::kCtl + Ctl::kMaskRing + 8 * (u & 31)) = mask;
      if (p.use_tma) {
        const uint32_t any = (mask | (mask >> 1) | (mask >> 2) | (mask >> 3)) & 0x11111111u;
        if (lane == 0) mbar_arrive_tx(full, static_cast<uint32_t>(__popc(any)) * 4u * row_pad);
        const int32_t row = val ? static_cast<int32_t>(pg0 * rows_per_page + in_page(pos0)) : 0;
        const int g = lane & 7;
        const uint32_t m4 = (mask >> (4 * g)) & 15u;
        const int first = m4 != 0u ? 4 * g + __ffs(m4) - 1 : 0;
        int32_t y[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
          y[k] = __shfl_sync(0xffffffffu, row, ((m4 >> k) & 1u) ? 4 * g + k : first);
        if (lane < kSub / 4 && m4 != 0u)
          gather4(raw_row(s, 4 * lane), tmap, y[0], y[1], y[2], y[3], full);
      } else {
        if (lane == 0) mbar_arrive_tx(full, static_cast<uint32_t>(__popc(mask)) * copy);
        __syncwarp();
        if (val) {
          const int64_t off = pg0 * p.block_stride + static_cast<int64_t>(in_page(pos0)) * L::kRowBytes;
          bulk_g2s(raw_row(s, lane), p.cache + off, copy, full);
        }
      }
      __syncwarp();
      if (lane == 0)
        st_shared_u32(ctl + Ctl::kLastStage + 4 * (u % kRawBars), static_cast<uint32_t>(u + 1));
      pos0 = pos1;
      pos1 = pos2;
      pos2 = pos3;
      pos3 = pos4;
      pg0 = pg1;
      pg1 = pg2;
    }
  } else if (warp == kQWarp && rank == 0) {
    convert_q(128 + lane);
  } else if (warp >= kDequantWarp0 && rank == 0) {
    // ------------------------------------------------ score CTA: rows -> K chunks in TMEM
    // Warp (set, quadrant) = ((w - 8) / 4, w % 4) expands, for every tile i,
    // its share of the 32 rows of stage 4 i + quadrant into TMEM lanes
    // 32 quadrant .. + 31 (thread = row): set 0 the latent chunks 0 and 2
    // (dims 0..127, 256..383) and the rope (chunk 4), set 1 the latent chunks
    // 1 and 3. The MMA takes the chunks in order, so the two sets feed it in
    // turn and work side by side. A chunk goes into the next slot of the K
    // ring once the MMA has released it, in 64-dimension halves (32 columns
    // each; a half's store completes before its registers are reused); dead
    // rows are written as zeros. NVFP4 rows: each thread first loads its
    // whole share into registers and releases the gather stage, so a tile's
    // four stages never wait on one another.
    convert_q(160 + 32 * (warp - kDequantWarp0) + lane);
    const int quad = warp & 3;
    const int set = (warp - kDequantWarp0) >> 2;
    const uint32_t lane_base = static_cast<uint32_t>(32 * quad) << 16;
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
    bool run = true;
    for (int i = 0; i < n_tiles && run; ++i) {
      const int u = kPiecesPerTile * i + quad;
      const int s = u % L::kStagesS;   // data slot
      const int rb = u % kRawBars;     // barrier pair
      if (!warp_wait(bar(Ctl::kRawFull, rb), (u / kRawBars) & 1u, abort_addr, lim)) break;
      const bool ok = (mask_of(u) >> lane) & 1u;
      const uint32_t src = raw_row(s, lane);
      // the ring slot of chunk c of this tile, once the MMA has released it
      auto take_slot = [&](int c, uint32_t& col) -> bool {
        const int q = kChunksPerTile * i + c;
        const int cs = q % L::kKSlots;
        col = 64u * static_cast<uint32_t>(cs);
        if (!warp_wait(bar(Ctl::kChunkEmpty, cs), ((q / L::kKSlots) & 1u) ^ 1u, abort_addr, lim))
          return false;
        tc_fence_after();
        return true;
      };
      // 32 columns into TMEM, complete before the registers are reused
      auto put_half = [&](uint32_t c0, const uint32_t (&h)[32]) {
        tmem_st32(tmem + lane_base + c0, h);
        tmem_st_wait();
      };
      auto chunk_done = [&](int c) {
        const int cs = (kChunksPerTile * i + c) % L::kKSlots;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(Ctl::kChunkFull, cs));
      };
      uint32_t col = 0;
      if constexpr (L::kNv) {
        // Row reads stay within bytes [0, 352) of the row slot. Each set keeps
        // the codes of its two latent chunks (4 x 16 B each, at byte 64 c) and
        // their four scale words (words 2 c, 2 c + 1); set 0 also the rope
        // (4 x 16 B). The loop is rolled over the four 64-dimension halves
        // (one copy of the conversion code): each takes cw[0], cw[1] and
        // scw[0], then both shift.
        uint4 cw[8], rp[4];
        uint32_t scw[4];
        {
          const uint4 s0 = ok ? ld_shared_v4(src + kScaleOff) : z;
          const uint4 s1 = ok ? ld_shared_v4(src + kScaleOff + 16) : z;
          scw[0] = set == 0 ? s0.x : s0.z;
          scw[1] = set == 0 ? s0.y : s0.w;
          scw[2] = set == 0 ? s1.x : s1.z;
          scw[3] = set == 0 ? s1.y : s1.w;
        }
#pragma unroll
        for (int x = 0; x < 8; ++x)
          cw[x] = ok ? ld_shared_v4(src + 64u * (2u * (x >> 2) + set) + 16u * (x & 3)) : z;
#pragma unroll
        for (int x = 0; x < 4; ++x)
          rp[x] = (ok && set == 0) ? ld_shared_v4(src + kRopeOff + 16u * x) : z;
        uint32_t h[32];
#pragma unroll 1
        for (int j = 0; j < 4 && run; ++j) {
          const uint32_t w[8] = {cw[0].x, cw[0].y, cw[0].z, cw[0].w,
                                 cw[1].x, cw[1].y, cw[1].z, cw[1].w};
          nvfp4_chunk(w, scw[0], h);
          if (j == 0) {  // the share is in registers: the gather warp may refill the stage
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(Ctl::kRawEmpty, rb));
          }
          const int c = set + 2 * (j >> 1);  // chunk of this half
          if ((j & 1) == 0) run = take_slot(c, col);
          if (!run) break;
          put_half(col + 32u * static_cast<uint32_t>(j & 1), h);
          if (j & 1) chunk_done(c);
#pragma unroll
          for (int x = 0; x < 6; ++x) cw[x] = cw[x + 2];
#pragma unroll
          for (int x = 0; x < 3; ++x) scw[x] = scw[x + 1];
        }
        if (set == 0 && run) {  // the rope: chunk 4, 32 of its slot's columns
#pragma unroll
          for (int x = 0; x < 4; ++x) e4m3x16_to_f16(rp[x], h + 8 * x);
          run = take_slot(kChunksPerTile - 1, col);
          if (run) {
            put_half(col, h);
            chunk_done(kChunksPerTile - 1);
          }
        }
      } else {
        // FP8 rows: half by half from shared memory; set 0 the chunks 0, 2 and
        // the rope (bytes 512..575), set 1 the chunks 1 and 3; the stage is
        // released after the set's last read of it
        const int nhalf = set == 0 ? 5 : 4;
#pragma unroll 1
        for (int j = 0; j < nhalf && run; ++j) {
          const int c = j < 4 ? set + 2 * (j >> 1) : kChunksPerTile - 1;
          const uint32_t off = 128u * static_cast<uint32_t>(c) + 64u * static_cast<uint32_t>(j & 1);
          uint32_t h[32];
#pragma unroll
          for (int x = 0; x < 4; ++x)
            e4m3x16_to_f16(ok ? ld_shared_v4(src + off + 16 * x) : z, h + 8 * x);
          if (j == nhalf - 1) {
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(Ctl::kRawEmpty, rb));
          }
          if ((j & 1) == 0) run = take_slot(c, col);
          if (!run) break;
          put_half(col + 32u * static_cast<uint32_t>(j & 1), h);
          if ((j & 1) || j == 4) chunk_done(c);
        }
      }
    }
  } else if (warp >= kDequantWarp0) {
    // ------------------------------------------------ output CTA: gather + V slots
    // V (rows x 512 dims, FP16) is read by the P V MMA MN-major: each 32-row
    // slot holds 8 blocks of 64 dims, each block 4 groups of 8 rows x 128 B.
    const int dq = warp - kDequantWarp0;  // 0..7
    bool run = true;
    // V slot u % 3 is free once the P V MMAs of piece u - 3 have completed
    // (the one commit per piece, on its P buffer's PvDone barrier)
    auto v_slot_free = [&](int u) {
      if (u < L::kVSlots) return true;
      const int v = u - L::kVSlots;
      return warp_wait(bar(Ctl::kPvDone, v % kPBufs), (v / kPBufs) & 1u, abort_addr, lim);
    };
    for (int u = 0; u < n_pc && run; ++u) {
      const int s = u % L::kStagesO;   // data slot
      const int rb = u % kRawBars;     // barrier pair
      const int vs = u % L::kVSlots;
      if (!warp_wait(bar(Ctl::kRawFull, rb), (u / kRawBars) & 1u, abort_addr, lim)) break;
      const uint32_t mask = mask_of(u);
      const uint32_t vslot = sbase + vs * L::kVSlot;
      if constexpr (L::kNv) {
        // Items of 32 dims (16 code bytes + 2 scale bytes): lane = (jj & 1) +
        // 2 rr + 8 (jj >> 1) over 4 rows x 8 items, two items per thread; the
        // loads, the scale reads and the swizzled stores are conflict free.
        // The loads go out before the wait for the slot.
        uint4 cd[2];
        uint32_t scv[2];
        int rr[2], jj[2];
#pragma unroll
        for (int it = 0; it < 2; ++it) {
          const int blk = it * 8 + dq;
          rr[it] = 4 * (blk & 7) + ((lane >> 1) & 3);
          jj[it] = 8 * (blk >> 3) + (lane & 1) + 2 * (lane >> 3);
          const bool ok = (mask >> rr[it]) & 1u;
          const uint32_t rp = raw_row(s, rr[it]);
          cd[it] = ok ? ld_shared_v4(rp + 16 * jj[it]) : make_uint4(0u, 0u, 0u, 0u);
          scv[it] = ok ? ld_shared_u16(rp + kScaleOff + 2 * jj[it]) : 0u;
        }
        if (!v_slot_free(u)) break;
#pragma unroll
        for (int it = 0; it < 2; ++it) {
          const uint32_t s0 = scale_f16x2(scv[it]), s1 = scale_f16x2(scv[it] >> 8);
          const uint32_t w[4] = {cd[it].x, cd[it].y, cd[it].z, cd[it].w};
          uint32_t h[16];
#pragma unroll
          for (int x = 0; x < 4; ++x) {
            uint32_t f[4];
            e2m1x8_to_f16x8(w[x], f);
#pragma unroll
            for (int y = 0; y < 4; ++y) h[4 * x + y] = hmul2_u32(f[y], x < 2 ? s0 : s1);
          }
          const uint32_t blk = vslot + static_cast<uint32_t>(jj[it] >> 1) * 4096u;
          const uint32_t c0 = static_cast<uint32_t>((jj[it] & 1) * 4);
#pragma unroll
          for (int c = 0; c < 4; ++c)
            st_shared_v4(blk + sw128_off(static_cast<uint32_t>(rr[it]), c0 + c), h[4 * c],
                         h[4 * c + 1], h[4 * c + 2], h[4 * c + 3]);
        }
      } else {
        if (!v_slot_free(u)) break;
        const int dt = dq * 32 + lane;
#pragma unroll
        for (int it = 0; it < 4; ++it) {
          const int item = dt + 256 * it;
          const int r = item & 31;          // row within the slot
          const int j = item >> 5;          // 16-dim group 0..31
          const bool ok = (mask >> r) & 1u;
          uint32_t h[8];
          e4m3x16_to_f16(ok ? ld_shared_v4(raw_row(s, r) + 16 * j) : make_uint4(0u, 0u, 0u, 0u),
                         h);
          const uint32_t blk = vslot + (j >> 2) * 4096u;
          const uint32_t c0 = static_cast<uint32_t>((j & 3) * 2);
          st_shared_v4(blk + sw128_off(r, c0), h[0], h[1], h[2], h[3]);
          st_shared_v4(blk + sw128_off(r, c0 + 1), h[4], h[5], h[6], h[7]);
        }
      }
      fence_proxy_async_cta();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(bar(Ctl::kVtFull, vs));
        mbar_arrive(bar(Ctl::kRawEmpty, rb));  // stage u read: the gather warp may refill slot s
      }
    }
    epilogue(warp & 3, 1 + ((warp - kDequantWarp0) >> 2), 4 + (warp - kDequantWarp0));
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------ MMA issue (one thread)
    if (lane == 0) {
      uint32_t last_bar = 0, last_parity = 0;
      bool issued = false;
      if (rank == 0) {
        if (wait_bar_hot(bar(Ctl::kQReady, 0), 0, abort_addr, lim)) {
          // Operands from loop-invariant bases: the allocation of all 512
          // columns starts at TMEM address 0 (checked at set-up); a
          // descriptor's address field counts 16 bytes.
          const uint64_t qd = sw128_desc(sbase + L::kQ);
          const uint32_t idesc = idesc_qk(p.num_heads);
          bool run = true;
          // Whether chunk q is known to be in the ring: the next chunk's
          // barrier is tested (without blocking) before this chunk's MMAs go
          // out, so a chunk that is already there costs no wait at all.
          bool ready = false;
          for (int i = 0; i < n_tiles && run; ++i) {
            const int s2 = i % L::kSBufs;
            const uint32_t sph = static_cast<uint32_t>(i / L::kSBufs) & 1u;
            if (!wait_bar_hot(bar(Ctl::kSEmpty, s2), sph ^ 1u, abort_addr, lim)) break;
            const uint32_t dcol = L::kSCol + 128u * s2;
            for (int kb = 0; kb < kChunksPerTile; ++kb) {
              const int q = kChunksPerTile * i + kb;
              const int cs = q % L::kKSlots;
              if (!ready &&
                  !wait_bar_hot(bar(Ctl::kChunkFull, cs), (q / L::kKSlots) & 1u, abort_addr, lim)) {
                run = false;
                break;
              }
              tc_fence_after();
              ready = mbar_ready(bar(Ctl::kChunkFull, (q + 1) % L::kKSlots),
                                 ((q + 1) / L::kKSlots) & 1u);
              // chunk kb < 4: Q tiles 2 kb and 2 kb + 1 (8 MMAs); the rope: Q tile 8
              const uint64_t bd = qd + static_cast<uint64_t>(2 * kb * (L::kQTile >> 4));
              const uint32_t a = 64u * static_cast<uint32_t>(cs);
              const int nk = kb < kChunksPerTile - 1 ? 8 : 4;
#pragma unroll
              for (int kk = 0; kk < 8; ++kk)
                if (kk < nk)
                  mma_ts(dcol, a + 8u * kk,
                         bd + static_cast<uint64_t>((kk >> 2) * (L::kQTile >> 4) + 2 * (kk & 3)),
                         idesc, (kb | kk) != 0 ? 1u : 0u);
              mma_commit(bar(Ctl::kChunkEmpty, cs));
              last_bar = bar(Ctl::kChunkEmpty, cs);
              last_parity = (q / L::kKSlots) & 1u;
              issued = true;
            }
            if (run) mma_commit(bar(Ctl::kSFull, s2));
          }
        }
      } else {
        uint32_t n_corr = 0;
        // the next piece's P and V barriers are tested (without blocking)
        // before this piece's MMAs go out
        bool p_ready = false, v_ready = false;
        for (int u = 0; u < n_pc; ++u) {
          const int pb = u % kPBufs;
          const int vs = u % L::kVSlots;
          // P (and any rescale of O) first, then the V slot
          if (!p_ready &&
              !wait_bar_hot<true>(bar(Ctl::kPFull, pb), (u / kPBufs) & 1u, abort_addr, lim))
            break;
          const uint4 fl = ld_shared_v4(sbase + L::kAFO + pb * kAFBytes + 512);
          if ((fl.x | fl.y | fl.z | fl.w) != 0u) {
            if (!wait_bar_hot(bar(Ctl::kOCorr, 0), n_corr & 1u, abort_addr, lim)) break;
            ++n_corr;
          }
          if (!v_ready && !wait_bar_hot(bar(Ctl::kVtFull, vs), (u / L::kVSlots) & 1u, abort_addr, lim))
            break;
          tc_fence_after();
          p_ready = mbar_ready<true>(bar(Ctl::kPFull, (u + 1) % kPBufs), ((u + 1) / kPBufs) & 1u);
          v_ready = mbar_ready(bar(Ctl::kVtFull, (u + 1) % L::kVSlots), ((u + 1) / L::kVSlots) & 1u);
          const uint32_t pbuf = sbase + L::kP + pb * kPiece;
          const uint32_t vslot = sbase + vs * L::kVSlot;
#pragma unroll
          for (int kk = 0; kk < 2; ++kk) {
            const uint64_t adesc = sw128_desc_mn(pbuf + 2048u * kk);
#pragma unroll
            for (int nh = 0; nh < 2; ++nh) {
              const uint64_t bdesc = sw128_desc_mn(vslot + 2048u * kk + 16384u * nh);
              mma_ss(tmem + 256u * nh, adesc, bdesc, kIdescPV, (u > 0 || kk > 0) ? 1u : 0u);
            }
          }
          mma_commit(bar(Ctl::kPvDone, pb));  // frees P buffer pb and V slot vs
          last_bar = bar(Ctl::kPvDone, pb);  // tracks every MMA issued so far
          last_parity = (u / kPBufs) & 1u;
          issued = true;
        }
      }
      if (issued) drain_bar(last_bar, last_parity);  // every issued MMA has completed
    }
  } else if (warp < 4 && rank == 0) {
    // ------------------------------------------------ score CTA: Q set-up, then softmax
    const int q4 = warp;  // quadrant: rows 32 q4 .. + 31 of each tile
    const uint32_t lane_base = static_cast<uint32_t>(32 * q4) << 16;
    // `ok` is the same in the four warps (it changes only at their group
    // barriers, so they all pass the same barriers in the same order); `sent`
    // is this warp's own: whether its waits for the peer's P buffers held. A
    // warp whose wait ran out stores nothing more into the peer and follows
    // the others to the next group barrier, where they all stop.
    bool ok, sent = true;
    {
      // this warp's share of Q, then the initial reference maxima
      st_shared_u32(sbase + L::kNegM + 4 * tid, __float_as_uint(INFINITY));  // m_ref = -inf
      convert_q(tid);
      ok = group_and(ld_shared_u32(abort_addr) == 0u);  // also: every m_ref is initialised
    }
    const float c = p.score_scale;
    const uint64_t c2 = f32x2(c, c);
    const int hchunks = (p.num_heads + 31) >> 5;  // head chunks with live heads
    const uint32_t stg = sbase + L::kStg + q4 * kPiece;  // NVFP4 rows
    const uint32_t peer_p = map_rank(sbase + L::kP, peer);
    const uint32_t peer_af = map_rank(sbase + L::kAFO, peer);
    const uint32_t peer_ctl = map_rank(ctl, peer);
    // P^T of this warp's 32 rows for head chunk hc (32 heads) from S^T at
    // column `scol`, stored at `dst` (the staging slot, or the peer's P
    // buffer); returns the largest exponent t = s c - m_ref of a live row.
    auto p_chunk = [&](uint32_t scol, int hc, bool live, uint32_t dst) -> float {
      uint32_t sv[32];
      tmem_ld32(tmem + lane_base + scol + 32u * hc, sv);
      float nm[32];
#pragma unroll
      for (int v = 0; v < 8; ++v) {
        const uint4 x = ld_shared_v4(sbase + L::kNegM + 128 * hc + 16 * v);
        nm[4 * v] = __uint_as_float(x.x);
        nm[4 * v + 1] = __uint_as_float(x.y);
        nm[4 * v + 2] = __uint_as_float(x.z);
        nm[4 * v + 3] = __uint_as_float(x.w);
      }
      tmem_ld_wait();
      float tmx = -INFINITY;
      uint32_t pk[16];
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        float t0, t1;
        f32x2_split(fma_f32x2(f32x2(__uint_as_float(sv[2 * q]), __uint_as_float(sv[2 * q + 1])),
                              c2, f32x2(nm[2 * q], nm[2 * q + 1])),
                    t0, t1);
        tmx = fmax3(tmx, t0, t1);
        pk[q] = live ? pack_f16x2(ex2(t0), ex2(t1)) : 0u;
      }
      // heads 32 hc .. + 31 = M block hc / 2, 16-byte chunks 4 (hc % 2) .. + 3
      const uint32_t blk = dst + static_cast<uint32_t>(hc >> 1) * 4096u;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        const uint32_t a = blk + sw128_off(static_cast<uint32_t>(lane), 4 * (hc & 1) + cc);
        if constexpr (L::kDirectP) {
          if (sent) st_cluster_v4(a, pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3]);
        } else
          st_shared_v4(a, pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3]);
      }
      return live ? tmx : -INFINITY;
    };
    for (int i = 0; i < n_tiles && ok; ++i) {
      const int s2 = i % L::kSBufs;
      const uint32_t scol = L::kSCol + 128u * s2;
      ok = group_and(sent && wait_bar(bar(Ctl::kSFull, s2), (i / L::kSBufs) & 1u, abort_addr, lim));
      if (!ok) break;
      tc_fence_after();
      const int u = kPiecesPerTile * i + q4;
      const bool live = (mask_of(u) >> lane) & 1u;
      const int pb = u % kPBufs;
      uint32_t dst = stg;
      if constexpr (L::kDirectP) {
        // piece u is written straight into the peer's P buffer u % 6, once the
        // peer has released it
        uint32_t free_ok = 1u;
        if (lane == 0)
          free_ok = wait_bar<true>(bar(Ctl::kPEmpty, pb), ((u / kPBufs) & 1u) ^ 1u, abort_addr, lim)
                        ? 1u : 0u;
        sent = __shfl_sync(0xffffffffu, free_ok, 0) != 0u;
        dst = peer_p + static_cast<uint32_t>(pb) * kPiece;
      } else {
        // this warp's staging slot: its copy of the previous tile has read it
        if (lane == 0) bulk_wait_read<0>();
        __syncwarp();
      }
      // Pass 0 computes P against the current references. A live score above
      // its head's reference by more than tau (every first live score
      // included) moves the reference to the tile's maximum: all four warps
      // then take the rare path together and pass 1 recomputes P (one copy
      // of the P code for both passes).
      bool exceed = false;
#pragma unroll 1
      for (int pass = 0; pass < 2; ++pass) {
        float tmx = -INFINITY;
#pragma unroll 1
        for (int hc = 0; hc < hchunks; ++hc) tmx = fmaxf(tmx, p_chunk(scol, hc, live, dst));
        if (pass == 1) break;
        exceed = group_or(tmx > kTau);
        if (!exceed) break;
        // new reference maxima, their rescale factors and flags
        softmax_new_refs<L>(sbase, tmem + lane_base + scol, live, c, i > 0);
        ok = group_and(ok);  // new references, factors and flags are visible
        if (!ok) break;
      }
      if (!ok) break;
      // S^T buffer s2 is read: the MMA may overwrite it
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(Ctl::kSEmpty, s2));
      if constexpr (L::kDirectP) {
        if (!sent) continue;
        // factors (tile's first piece) or zero flags straight into the peer's
        // factor block; every lane releases its stores and arrives
        const uint32_t af = peer_af + static_cast<uint32_t>(pb) * kAFBytes;
        if (q4 == 0) {
          if (exceed) {
            const uint4 a = ld_shared_v4(sbase + L::kAlpha + 16 * lane);
            st_cluster_v4(af + 16 * lane, a.x, a.y, a.z, a.w);
          }
          if (lane == 0) {
            const uint4 f = exceed ? ld_shared_v4(sbase + L::kFlags) : make_uint4(0u, 0u, 0u, 0u);
            st_cluster_v4(af + 512, f.x, f.y, f.z, f.w);
          }
        } else if (lane == 0) {
          st_cluster_v4(af + 512, 0u, 0u, 0u, 0u);
        }
        fence_proxy_async_cluster();  // the peer's MMAs read P through the async proxy
        mbar_arrive_cluster(peer_ctl + Ctl::kPFull + 8 * pb);
        continue;
      }
      // rescale factors travel with the tile's first piece (slot 0); pieces
      // 1-3 carry zero flags
      if (q4 == 0) {
        if (exceed) {
          const uint4 a = ld_shared_v4(sbase + L::kAlpha + 16 * lane);
          st_shared_v4(sbase + L::kAFS + 16 * lane, a.x, a.y, a.z, a.w);
        }
        if (lane == 0) {
          const uint4 f = exceed ? ld_shared_v4(sbase + L::kFlags) : make_uint4(0u, 0u, 0u, 0u);
          st_shared_v4(sbase + L::kAFS + 512, f.x, f.y, f.z, f.w);
        }
      } else if (lane == 0) {
        st_shared_v4(sbase + L::kAFS + kAFBytes + (q4 - 1) * kFlagBytes, 0u, 0u, 0u, 0u);
      }
      fence_proxy_async_cta();  // generic stores -> visible to the bulk copies
      __syncwarp();
      // Piece u goes into the peer's P buffer u % 6 once the peer has released
      // it, with the rescale factors (tile's first piece) or zero flags.
      uint32_t sent_ok = 1u;
      if (lane == 0) {
        sent_ok = wait_bar<true>(bar(Ctl::kPEmpty, pb), ((u / kPBufs) & 1u) ^ 1u, abort_addr, lim)
                      ? 1u : 0u;
        if (sent_ok) {
          const uint32_t fb = q4 == 0 ? kAFBytes : kFlagBytes;
          const uint32_t src_af = q4 == 0 ? sbase + L::kAFS
                                          : sbase + L::kAFS + kAFBytes + (q4 - 1) * kFlagBytes;
          const uint32_t pbar = peer_ctl + Ctl::kPFull + 8 * pb;
          mbar_arrive_tx_cluster(pbar, kPiece + fb);
          bulk_s2s(peer_p + pb * kPiece, stg, kPiece, pbar);
          // flags land at byte 512 of the buffer's factor block
          bulk_s2s(peer_af + pb * kAFBytes + (q4 == 0 ? 0u : 512u), src_af, fb, pbar);
          bulk_commit();
          st_shared_u32(ctl + Ctl::kSentCnt + 4 * pb, static_cast<uint32_t>(u / kPBufs + 1));
        }
      }
      sent = __shfl_sync(0xffffffffu, sent_ok, 0) != 0u;
    }
    if (lane == 0) bulk_wait_read<0>();  // every copy has read this warp's slot
    ok = group_and(ok && sent);
    // the peer learns how many pieces went into each P buffer (it drains them
    // on abort), then the final reference maximum of head h = tid
    if (tid == 0 && !L::kDirectP) {
#pragma unroll
      for (int pb = 0; pb < kPBufs; ++pb)
        st_cluster_u32(peer_ctl + Ctl::kSent + 4 * pb, ld_shared_u32(ctl + Ctl::kSentCnt + 4 * pb));
      mbar_arrive_cluster(peer_ctl + Ctl::kSentBar);
    }
    if (ok) {
      const float m = -__uint_as_float(ld_shared_u32(sbase + L::kNegM + 4 * tid));
      st_cluster_u32(map_rank(sbase + L::kFinO, peer) + 4 * tid, __float_as_uint(m));
      mbar_arrive_cluster(peer_ctl + Ctl::kStats);
    }
  } else if (warp < 4) {
    // ------------------------------------------------ output CTA: corrections + epilogue
    // Per piece u (thread = head h): a rescale of O and l when the piece's
    // flags say the score CTA raised its reference maximum (the previous
    // piece's MMAs are complete by then), then the sum of P^T column h of the
    // piece into l, then, once the piece's MMAs are complete, the P buffer goes
    // back to the score CTA.
    const int h = warp * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t peer_ctl = map_rank(ctl, peer);
    // column h of a P^T piece: M block h / 64, 16-byte chunk (h % 64) / 8
    const uint32_t col_blk = static_cast<uint32_t>(h >> 6) * 4096u + (static_cast<uint32_t>(h) & 7u) * 2u;
    const uint32_t col_chunk = (static_cast<uint32_t>(h) & 63u) >> 3;
    // byte offset of row r of that column: (r / 8) 1024 + xo[r % 8]
    uint32_t xo[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) xo[k] = col_blk + sw128_off(static_cast<uint32_t>(k), col_chunk);
    float l_acc = 0.f;
    bool ok = true;
    for (int u = 0; u < n_pc; ++u) {
      const int pb = u % kPBufs;
      if (!warp_wait<true>(bar(Ctl::kPFull, pb), (u / kPBufs) & 1u, abort_addr, lim)) {
        ok = false;
        break;
      }
      const uint32_t afp = sbase + L::kAFO + pb * kAFBytes;
      const uint4 fl = ld_shared_v4(afp + 512);
      if ((fl.x | fl.y | fl.z | fl.w) != 0u) {
        const float alpha = __uint_as_float(ld_shared_u32(afp + 4 * h));
        l_acc *= alpha;
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
      const uint32_t pbase = sbase + L::kP + pb * kPiece;
      float part[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int r = 0; r < kSub; ++r)
        part[r & 3] += f16_bits_to_f32(static_cast<uint16_t>(
            ld_shared_u16(pbase + xo[r & 7] + static_cast<uint32_t>(r >> 3) * 1024u)));
      l_acc += (part[0] + part[1]) + (part[2] + part[3]);
      if (!warp_wait(bar(Ctl::kPvDone, pb), (u / kPBufs) & 1u, abort_addr, lim)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // this warp has read buffer pb (flags, factors, column sums) and its
      // MMAs are done: the score CTA may refill it
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster_relaxed(peer_ctl + Ctl::kPEmpty + 8 * pb);
    }
    float m_fin = NAN, l_fin = l_acc;
    ok = __all_sync(0xffffffffu, ok);
    if (ok && warp_wait<true>(bar(Ctl::kStats, 0), 0, abort_addr, lim)) {
      m_fin = __uint_as_float(ld_shared_u32(sbase + L::kFinO + 4 * h));
    } else {
      ok = false;
    }
    ok = group_and(ok);  // the four correction warps agree
    {
      const bool live = h < p.num_heads;
      const float inv = !ok ? NAN : (l_fin > 0.f ? 1.f / l_fin : 0.f);
      const float lse_nat = !ok ? NAN : (l_fin > 0.f ? (m_fin + lg2(l_fin)) * kLn2 : -INFINITY);
      const int64_t qh = static_cast<int64_t>(t) * p.num_heads + h;
      const bool single = p.num_splits == 1;
      const int64_t part = (static_cast<int64_t>(t) * p.num_splits + split) * p.num_heads + h;
      const bool f32 = !(single && !p.out_fp32);
      st_shared_u32(sbase + L::kScO + 4 * h, __float_as_uint(single ? inv * p.out_mult : inv));
      if (tid == 0) st_shared_u32(sbase + L::kEpiOk, ok ? 1u : 0u);
      if (!ok && live) {
        // a failed unit: NaN straight to global memory (its shared memory may
        // still receive copies, drained at teardown)
#pragma unroll 1
        for (int d = 0; d < kLatent; d += 4) {
          if (!f32)
            *reinterpret_cast<uint2*>(static_cast<uint16_t*>(p.out) + qh * kLatent + d) =
                make_uint2(pack_bf16x2(NAN, NAN), pack_bf16x2(NAN, NAN));
          else if (single)
            *reinterpret_cast<float4*>(static_cast<float*>(p.out) + qh * kLatent + d) =
                make_float4(NAN, NAN, NAN, NAN);
          else
            *reinterpret_cast<float4*>(p.ws + part * kLatent + d) =
                make_float4(NAN, NAN, NAN, NAN);
        }
      }
      epilogue(warp, 0, warp);
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
  if (tid == 0 && ld_shared_u32(abort_addr) != 0) {
    // A unit that gave up may still have copies in flight into this CTA's
    // shared memory: wait (bounded, ignoring the abort flag) for the last
    // phase of every gather stage that was armed and issued, for the Q copies,
    // and (output CTA) for every P piece the peer sent.
    for (int s = 0; s < kRawBars; ++s) {
      const uint32_t lu = ld_shared_u32(ctl + Ctl::kLastStage + 4 * s);
      if (lu > 0) drain_bar(bar(Ctl::kRawFull, s), ((lu - 1) / kRawBars) & 1u);
    }
    if (rank == 0) drain_bar(bar(Ctl::kQFull, 0), 0);
    if (rank == 1 && !L::kDirectP) {  // P copies (stored P is ordered by the cluster barrier)
      drain_bar<true>(bar(Ctl::kSentBar, 0), 0);
      for (int pb = 0; pb < kPBufs; ++pb) {  // pieces go into a buffer in order
        const uint32_t c = ld_shared_u32(ctl + Ctl::kSent + 4 * pb);
        if (c > 0) drain_bar<true>(bar(Ctl::kPFull, pb), (c - 1) & 1u);
      }
    }
  }
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
      // score rows: whole rows; output rows: the latent part (FP8: + 16 bytes)
      const cuuint32_t box_s[2] = {static_cast<cuuint32_t>(L::kRowS / L::kElem), 1};
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

// q_latent [num_q * H, 512] and q_rope [num_q * H, 64] bf16 as 2-D tensors
// with (heads rounded up to 8)-row x 64-column boxes in the 128-byte swizzle
// the MMA reads.
bool q_maps(const DecodeParams& p, CUtensorMap* ml, CUtensorMap* mr) {
  EncodeTiledFn enc = encode_tiled();
  const int64_t rows = static_cast<int64_t>(p.num_q) * p.num_heads;
  if (enc == nullptr || rows <= 0 || rows > 0x7FFFFFFFll) return false;
  const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(q_rows(p.num_heads))};
  const cuuint32_t es[2] = {1, 1};
  const cuuint64_t dl[2] = {static_cast<cuuint64_t>(kLatent), static_cast<cuuint64_t>(rows)};
  const cuuint64_t sl[1] = {static_cast<cuuint64_t>(kLatent * 2)};
  const cuuint64_t dr[2] = {static_cast<cuuint64_t>(kRope), static_cast<cuuint64_t>(rows)};
  const cuuint64_t sr[1] = {static_cast<cuuint64_t>(kRope * 2)};
  return enc(ml, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(p.q_lat), dl, sl, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
             CUDA_SUCCESS &&
         enc(mr, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(p.q_rope), dr, sr, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
             CUDA_SUCCESS;
}

template <int kFmt>
int32_t launch_fmt(const DecodeParams& p, cudaStream_t stream) {
  constexpr int smem = TcLayout<kFmt>::kBytes;
  cudaFuncSetAttribute(decode_tc_kernel<kFmt>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  const int64_t ctas = 2ll * p.num_q * p.num_splits;
  if (ctas > 0x7FFFFFFF) return NVFP4_MLA_ERR_SHAPE;
  DecodeParams q = p;
  CUtensorMap ms, mo, ml, mr;
  memset(&ms, 0, sizeof(ms));
  memset(&mo, 0, sizeof(mo));
  if (!q_maps(p, &ml, &mr)) return NVFP4_MLA_ERR_LAUNCH;
  q.use_tma = row_maps<kFmt>(p, &ms, &mo) ? 1 : 0;
  decode_tc_kernel<kFmt><<<static_cast<unsigned>(ctas), kThreads, smem, stream>>>(q, ms, mo, ml,
                                                                                   mr);
  return launch_status();
}

}  // namespace

int32_t launch_decode_tc(const DecodeParams& p, int row_format, cudaStream_t stream) {
  if (row_format == NVFP4_MLA_ROW_FP8_576) return launch_fmt<NVFP4_MLA_ROW_FP8_576>(p, stream);
  return launch_fmt<NVFP4_MLA_ROW_NVFP4_352>(p, stream);
}

}  // namespace nvfp4_mla
