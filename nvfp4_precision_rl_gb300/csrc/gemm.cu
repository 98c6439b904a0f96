// gemm.cu -- block-scaled W4A4 GEMMs on the sm_103a tensor cores (tcgen05).
//
//   Y[m, n] = bf16_rn( S_a[m] * S_b[n] * sum_k dec(a)[m, k] * dec(b)[n, k] )
//
// dec(.) = E4M3 block scale x E2M1 value; the block scales are applied by the
// tensor core itself (tcgen05.mma kind::mxf4nvf4, block_scale, 4 scales per
// 64-element K step) and the per-token / per-row FP32 scales in the epilogue, in
// the same kernel ("Towards Blackwell-Native 8-bit and 4-bit RL", results item
// 10: applying the per-token scale as a separate op is what made the unfused
// path slower than BF16; "TRIAGE", section "NVFP4 quantization format and W4A4
// execution": W4A4 runs natively on the tensor cores).
//
// Both GEMMs run on two-SM clusters (tcgen05 cta_group::2): the even CTA of a
// pair issues M = 256, N = 256 MMAs whose A rows come from both CTAs' shared
// memory (128 each) and whose 256 B rows are split 128/128 between them; each
// CTA holds its own 128 x 256 FP32 accumulator in TMEM.  Persistent: one pair
// per two SMs, tiles strided over the pairs.  Per CTA, warp-specialised:
//   warp 0 / warp 2  TMA producers (A and its scales / this CTA's B rows and
//               the B scales) into a 5-stage shared-memory ring; two issuing
//               threads because one thread's TMA copies are processed serially.
//   warp 1      TMEM allocation (collective across the pair); in the even CTA
//               the MMA issuer: warp-uniform loop, one elected lane issues the
//               MMAs and the multicast commits that release both CTAs' stages.
//   warps 4..7  scale warps, one per TMEM lane quadrant: each reads the stage's
//               512-byte scale atoms from shared memory (line = lane) and writes
//               them into its own 32 TMEM lanes with tcgen05.st -- the same
//               4-way replicated image a tcgen05.cp 32x128b.warpx4 would make,
//               but on the warps' TMEM store path, which (measured) overlaps the
//               MMAs, whereas every tcgen05.cp occupies the serial MMA pipe --
//               then arrive on the even CTA's barrier.
//   warps 8..15 epilogue, two warps per TMEM lane quadrant (128 columns each):
//               tcgen05.ld all 128 columns in one round, release the
//               accumulator, then scale by S_a * S_b with packed FP32x2
//               multiplies, round to bf16, stage in 128-byte swizzled shared
//               memory and store with TMA.  setmaxnreg moves registers from the
//               producer / MMA and scale warpgroups (64 and 80 per thread) to
//               the epilogue warpgroups (184), which hold the 128 columns.
// Tile 256 x 256 per pair, K step of 256 FP4 = 128 bytes = one swizzle row.
// The grouped (MoE) variant walks the padded per-expert layout (device-side
// offsets): a pair tile covers 256 rows of one expert -- with 128-row aligned
// segments it starts at every second 128-row tile of an expert (an odd tail
// computes, and drops, 128 rows past the expert), with 256-row aligned
// segments every 256-row slot is a pair tile.
//
// Every wait is bounded: a wait that runs out sets the status word and a shared
// abort flag, every role leaves its loop, the producers wait (bounded) for their
// copies in flight, the MMA warp for its tensor-core work, and TMEM is freed.
// (The scale warps' tcgen05.st are complete before they signal, so they leave
// nothing in flight.)
#include <cuda.h>

#include <atomic>

#include "common.cuh"
#include "swiglu.cuh"

namespace nvfp4 {
namespace {

constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kBKBytes = 128;                // 256 FP4 values per K step
constexpr int kMmaPerStage = 4;              // K = 64 per tcgen05.mma
constexpr int kSFWarps = 4;                  // one per TMEM lane quadrant
constexpr int kEpiWarps = 8;                 // two per TMEM lane quadrant, 128 columns each
// Warp roles, aligned to warpgroups (setmaxnreg acts per warpgroup):
//   warpgroup 0: warp 0 A producer, warp 1 TMEM allocation + MMA issuer (even
//                CTA), warp 2 B producer, warp 3 the grouped epilogue's tile
//                scheduler (idle in the dense GEMM);
//   warpgroup 1: warps 4..7 scale warps; warpgroups 2 and 3: epilogue.
constexpr int kPBWarp = 2;                   // the B-side producer
constexpr int kSchedWarp = 3;                // the epilogue's tile scheduler
constexpr int kFirstSFWarp = 4;
constexpr int kFirstEpiWarp = kFirstSFWarp + kSFWarps;
constexpr uint32_t kATileBytes = kBM * kBKBytes;      // 16 KB
constexpr uint32_t kSFAtomBytes = 512;                // 128 rows x 4 scales
constexpr uint32_t kSFATileBytes = 4 * kSFAtomBytes;  // 2 KB per stage
constexpr uint32_t kSFBTileBytes = 8 * kSFAtomBytes;  // 4 KB per stage
// The swizzled scale arrays are read through 5D tensor maps
// [experts][halves][128-row tiles][2 kgroups rows][256 bytes]: 8 rows of 256
// bytes are the 4 atoms (2 KB) of one K step of one 128-row tile; a B box
// takes two tiles (consecutive, or with SwiGLU the gate and the up tile).
constexpr uint32_t kSFMapRowBytes = 256;
constexpr uint32_t kSFMapBoxRows = kSFATileBytes / kSFMapRowBytes;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSFTmemCol = 256;                  // after the 256 accumulator columns
constexpr uint32_t kSFTmemPerStage = 48;              // 16 (A) + 32 (B)
// Grouped GEMM: tile information for the epilogue, prepared one tile ahead by
// the scheduler warp: the tile's origin, whether this CTA stores, this CTA's
// 128 row scales S_a and the tile's 256 column scales S_b.  (The dense
// epilogue finds its tile arithmetically and loads its scales itself, into a
// per-warp copy of its S_b half in the same space.)
struct EpiInfo {
    int64_t m_base;
    int64_t n0;
    int32_t write;
    int32_t end;       // 1: no more tiles for this pair
    int32_t pad[2];
    float sa[128];
    float sb[kBN];
};
constexpr int kInfoSlots = 2;
constexpr uint32_t kSBBytes = kInfoSlots * sizeof(EpiInfo) > kEpiWarps * (kBN / 2) * 4
                                  ? kInfoSlots * sizeof(EpiInfo) : kEpiWarps * (kBN / 2) * 4;
// The grouped kernel keeps a copy of the expert offsets in the rest of that space.
constexpr int kSmemOffsets = static_cast<int>((kSBBytes - kInfoSlots * sizeof(EpiInfo)) / sizeof(int32_t));
static_assert(kSmemOffsets >= 129, "room for the offsets of 128 experts");
constexpr uint64_t kWaitLimitNs = 2000000000ull;      // 2 s: the default pipeline wait limit
constexpr uint64_t kDrainLimitNs = 50000000ull;       // 50 ms

struct GemmParams {
    const uint8_t* sfa;
    const uint8_t* sfb;
    const float* sa;
    const float* sb;
    uint16_t* y;
    const int32_t* offsets;   // grouped only
    unsigned* status;
    int64_t M;                // rows of A (dense) or rows capacity (grouped)
    int64_t N;
    int64_t ld_y;
    int64_t sfb_expert_bytes; // grouped: bytes of one expert's scale block
    int kgroups;              // K / 64: scale words per row
    int num_k_tiles;
    int num_n_tiles;
    int num_m_tiles;          // dense: ceil(M / 128); grouped: capacity tiles
    int E;                    // grouped: experts; dense: 0
    int sa_stride;            // 1: S_a per row of A; 0: one S_a for all rows
    int sb_stride;            // 1: S_b per row of B; 0: one S_b for all rows
    int n_fast;               // dense: 1 walks the tiles n-tile fastest, 0 m-tile fastest
    // Grouped SwiGLU epilogue (fc1 of a SwiGLU expert): B holds each expert's
    // F gate rows then its F up rows; a pair tile pairs gate rows n0 .. n0+127
    // (even CTA) with up rows F+n0 .. (odd CTA), and its epilogue writes
    // h = bf16(silu(g) u) for output columns n0 .. n0+127 of H [rows, F].
    int swiglu;               // 0 or 1
    int64_t ffn;              // swiglu: F (= N, the output columns)
    int64_t b_rows;           // rows of B per expert: N, or 2F with swiglu
    int n_step;               // output columns per tile: 256, or 128 with swiglu
    uint64_t wait_limit_ns;   // every pipeline wait gives up after this long
};

// ----------------------------------------------------------------------------
// PTX wrappers
// ----------------------------------------------------------------------------
__device__ __forceinline__ void tma_load_2d(const CUtensorMap* map, uint64_t* bar, void* dst,
                                            int32_t c0, int32_t c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];"
        ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0),
          "r"(c1)
        : "memory");
}

__device__ __forceinline__ void tma_load_5d(const CUtensorMap* map, uint64_t* bar, void* dst, int32_t c0,
                                            int32_t c1, int32_t c2, int32_t c3, int32_t c4) {
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6, %7}], [%2];"
        ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0),
          "r"(c1), "r"(c2), "r"(c3), "r"(c4)
        : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart (SBO), descriptor version 1.
__device__ __forceinline__ uint64_t sw128_desc(const void* p) {
    const uint64_t addr = smem_u32(p);
    return ((addr >> 4) & 0x3FFFull) | (1ull << 16) | ((1024ull >> 4) << 32) | (1ull << 46) |
           (2ull << 61);
}

// 32 lanes x 32 consecutive 32-bit columns; thread t gets lane (base + t).
// The registers are valid only after tmem_wait() on the same array, which
// follows immediately.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

// Wait for this thread's outstanding tcgen05.ld; naming the registers keeps
// every use of them below the wait.
__device__ __forceinline__ void tmem_wait(uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.wait::ld.sync.aligned;"
        : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
          "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),
          "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]),
          "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]),
          "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31]));
}

// Write 16 / 32 consecutive TMEM columns of this warp's 32 lanes.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};"
        ::"r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]),
          "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]),
          "r"(v[14]), "r"(v[15])
        : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};"
        ::"r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]),
          "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]),
          "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]),
          "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]),
          "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
        : "memory");
}

__device__ __forceinline__ void tmem_st_wait() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 32 accumulator columns -> 16 packed bf16 pairs: y = bf16_rn(acc * S_b[n] * S_a).
__device__ __forceinline__ void scale_chunk(const uint32_t (&r)[32], const float* sb, float sa,
                                            uint32_t* out) {
    const float2 sa2 = make_float2(sa, sa);
#pragma unroll
    for (int j = 0; j < 32; j += 4) {
        const float4 b4 = *reinterpret_cast<const float4*>(sb + j);
        float2 v0 = __fmul2_rn(make_float2(__uint_as_float(r[j]), __uint_as_float(r[j + 1])),
                               make_float2(b4.x, b4.y));
        float2 v1 = __fmul2_rn(make_float2(__uint_as_float(r[j + 2]), __uint_as_float(r[j + 3])),
                               make_float2(b4.z, b4.w));
        v0 = __fmul2_rn(v0, sa2);
        v1 = __fmul2_rn(v1, sa2);
        const __nv_bfloat162 h0 = __floats2bfloat162_rn(v0.x, v0.y);
        const __nv_bfloat162 h1 = __floats2bfloat162_rn(v1.x, v1.y);
        out[j / 2] = *reinterpret_cast<const uint32_t*>(&h0);
        out[j / 2 + 1] = *reinterpret_cast<const uint32_t*>(&h1);
    }
}

// Keeps the compiler from reading `r` before the preceding tcgen05.wait::ld.
__device__ __forceinline__ void reg_fence(uint32_t (&r)[32]) {
    asm volatile(""
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
                   "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]),
                   "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]),
                   "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]),
                   "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]),
                   "+r"(r[31]));
}

// TMA store of one box of Y from shared memory (bulk-group completion).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int32_t x, int32_t y) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];"
                 ::"l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(src)), "r"(x), "r"(y)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// the shared-memory source of every committed store has been read
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// every committed store has completed
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ----------------------------------------------------------------------------
// The pair kernel (tcgen05 cta_group::2)
// ----------------------------------------------------------------------------
// Each CTA stages its own 128 rows of A and one 128-row half of the B tile, so
// per SM each 256-deep K step moves 32 KB of operands into shared memory
// instead of the 48 KB a single-SM 128 x 256 tile needs.  Each CTA keeps its
// accumulator and the scale factors of its own MMA rows (A) and of all 256 B
// rows in its own TMEM, written by its own scale warps.  Cross-CTA signals:
//   scale warps (both CTAs) -> sf_ready of the even CTA (remote mbarrier arrive),
//   MMA commits            -> empty / acc_full of both CTAs (multicast commit),
//   epilogue (both CTAs)   -> acc_empty of the even CTA (remote arrive).
// Within each CTA of the grouped kernel the scheduler warp and the epilogue
// warps hand the tile-information ring back and forth through info_full /
// info_empty (local arrivals).
constexpr int kPStages = 5;
constexpr int kPThreads = 32 * (kFirstEpiWarp + kEpiWarps);       // 512
// Registers per thread after the split: the CTA launches with 128 per thread
// (65,536 in all); warpgroups 0 and 1 give theirs up so the epilogue warps can
// hold a whole 128-column half of the accumulator.  The sum must stay within
// the launch's total, or setmaxnreg.inc would wait for registers forever.
constexpr int kRegsLaunch = 128;
constexpr int kRegsWG0 = 64;
constexpr int kRegsWG1 = 80;
constexpr int kRegsEpi = 184;
// The SwiGLU epilogue holds fewer accumulator registers (it pairs 64 gate with
// 64 up columns) and its tile scheduler more index arithmetic: 80 / 80 / 168.
constexpr int kRegsWG0Swi = 80;
constexpr int kRegsWG1Swi = 80;
constexpr int kRegsEpiSwi = 168;
static_assert(128 * kRegsWG0Swi + 128 * kRegsWG1Swi + 256 * kRegsEpiSwi <= kPThreads * kRegsLaunch,
              "register split exceeds the launch's registers");
static_assert(kPThreads == 512, "four warpgroups");
static_assert(128 * kRegsWG0 + 128 * kRegsWG1 + 256 * kRegsEpi <= kPThreads * kRegsLaunch,
              "register split exceeds the launch's registers");
static_assert(kRegsWG0 % 8 == 0 && kRegsWG1 % 8 == 0 && kRegsEpi % 8 == 0, "setmaxnreg granularity");
constexpr int kPLoadLanes = 1;                                    // issuing lanes per producer warp
constexpr unsigned kPLoadMask = (1u << kPLoadLanes) - 1;
constexpr int kPBoxRows = 128 / kPLoadLanes;                      // rows of A or B per TMA box
constexpr uint32_t kPBHalfBytes = 128 * kBKBytes;                 // 16 KB
// Output staging: per epilogue warp one 32-row x 64-column bf16 box (4 KB),
// 128-byte swizzled so the tensor-map store reads it back in rows.
constexpr uint32_t kPOutBoxBytes = 32 * 128;
constexpr uint32_t kPOutBytes = kEpiWarps * kPOutBoxBytes;        // 32 KB
constexpr uint32_t kPCarveBytes = kPStages * (kATileBytes + kPBHalfBytes + kSFATileBytes + kSFBTileBytes) +
                                  kPOutBytes + kSBBytes + 256;
constexpr size_t kPSmemBytes = 232448;                            // the opt-in maximum (227 KB)
static_assert(kPCarveBytes + 512 <= kPSmemBytes, "shared memory carve-up");
// Instruction descriptor, kind::mxf4nvf4: A and B E2M1 (format 1 at bits 7 and
// 10), K-major, N = 256 (N >> 3 at bit 17), M = 256 across the pair (M >> 4 at
// bit 24), scales UE4M3 (bit 23 clear), scale-factor ids 0, dense.
constexpr uint32_t kPInstrDesc = (1u << 7) | (1u << 10) | ((256u >> 3) << 17) | ((256u >> 4) << 24);
static_assert(kSFTmemCol + kPStages * kSFTmemPerStage <= kTmemCols, "TMEM columns");

// true in exactly one active lane of the warp (all lanes must be converged)
__device__ __forceinline__ bool elect_one() {
    uint32_t pred;
    asm volatile("{\n\t.reg .pred P;\n\telect.sync _|P, %1;\n\tselp.b32 %0, 1, 0, P;\n\t}"
                 : "=r"(pred) : "r"(0xFFFFFFFFu));
    return pred != 0;
}

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// shared::cluster address of the same object in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t peer_addr(const void* p, uint32_t rank) {
    uint32_t out;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(smem_u32(p)), "r"(rank));
    return out;
}

// Arrive on a barrier named by its shared::cluster address (possibly the peer's).
// Default (CTA-scope release) semantics: what the arrival publishes is either
// tcgen05 work already completed by tcgen05.wait, or nothing.  (A cluster-scope
// release measured about 0.8 us per arrival here and held the scale warps to
// one stage per microsecond.)
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    return ok != 0;
}

__device__ __forceinline__ bool mbar_try_wait_cluster_hint(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns) : "memory");
    return ok != 0;
}

// The same wait for short (debug) limits, as mbar_wait_short.
__device__ __forceinline__ bool mbar_wait_cluster_short(uint64_t* bar, uint32_t parity, uint64_t limit_ns,
                                                        volatile int* abort) {
    const uint32_t hint = static_cast<uint32_t>(limit_ns / 10 + 1);
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        if (mbar_try_wait_cluster_hint(bar, parity, hint)) return true;
        if (global_timer_ns() - t0 > limit_ns) return false;
        if (abort != nullptr && *abort) return false;
    }
}

// Bounded wait with cluster-scope acquire (the arrivals come from the peer CTA).
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity, uint64_t limit_ns,
                                                  volatile int* abort) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait_cluster(bar, parity)) return true;
        if ((it & 63u) == 0u) {
            if (abort != nullptr && *abort) return false;
            if (global_timer_ns() - t0 > limit_ns) return false;
        }
    }
}

__device__ __forceinline__ void tc_commit_pair(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 ::"r"(smem_u32(bar)) : "memory");
}

// arrive on the barrier at this offset in both CTAs of the pair
__device__ __forceinline__ void tc_commit_pair_both(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(smem_u32(bar)), "h"(static_cast<uint16_t>(3))
        : "memory");
}

__device__ __forceinline__ void tc_mma_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                            uint32_t accumulate, uint32_t sfa_tmem, uint32_t sfb_tmem) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X"
        " [%0], %1, %2, %3, [%5], [%6], p;\n\t}"
        ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(kPInstrDesc), "r"(accumulate), "r"(sfa_tmem),
          "r"(sfb_tmem)
        : "memory");
}

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
                 ::: "memory");
}

// One 256 x 256 output tile of a CTA pair.
struct PairTile {
    bool run;          // grouped: false for a slot that does not start a pair tile
    int64_t m_base;    // first row of the pair; CTA r owns rows m_base + 128 r ..
    int64_t n0;        // first output column
    int64_t b_row0;    // first row of B in the (stacked) weights
    int64_t row_end;   // rows at or past this are not written: M, or the expert's end
    int expert;
};

// Dense: t -> (m-tile, n-tile), the smaller operand's tile index fastest, so
// the pairs working at one time share the larger operand's rows and that
// operand streams from HBM once while the smaller one stays in L2 (with m
// fastest at M = 65,536, N = 6,144 every n-tile would sweep all 67 MB of A
// again while the bf16 output pushes it out of L2).  Grouped: t -> (128-row tile g of
// the padded layout, n-tile), n fastest; a pair tile starts at every second
// 128-row tile of an expert's segment, so an expert with an odd number of
// tiles ends in a tile whose odd CTA reads rows past the expert (its results
// are computed with this expert's B and never stored).
template <bool kGrouped, bool kSwiGLU>
__device__ __forceinline__ PairTile pair_tile_at(const GemmParams& p, int t, int num_pm, int mrows,
                                                 const int32_t* offs = nullptr) {
    PairTile tl;
    if (!kGrouped) {
        const int mt = p.n_fast ? t / p.num_n_tiles : t % num_pm;
        const int nt = p.n_fast ? t % p.num_n_tiles : t / num_pm;
        tl.run = true;
        tl.m_base = static_cast<int64_t>(mt) * 256;
        tl.n0 = static_cast<int64_t>(nt) * kBN;
        tl.b_row0 = tl.n0;
        tl.row_end = p.M;
        tl.expert = 0;
        return tl;
    }
    const int nt = t % p.num_n_tiles;
    const int64_t m0 = static_cast<int64_t>(t / p.num_n_tiles) * mrows;
    const int64_t n0 = static_cast<int64_t>(nt) * (kSwiGLU ? 128 : kBN);
    // The last expert e with offsets[e] <= m0 (empty experts are passed over),
    // i.e. (the number of e < E with offsets[e] <= m0) - 1 for nondecreasing
    // offsets, found in two rounds of independent loads -- the first entry of
    // each block of 16 experts, then the block's entries -- rather than a
    // binary search's chain of dependent loads (each an L2 round trip here).
    const int nblk = (p.E + 15) >> 4;
    int cnt = 0;
    for (int b0 = 0; b0 < nblk; b0 += 8) {
        int v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = (b0 + j < nblk) ? offs[16 * (b0 + j)] : INT_MAX;
#pragma unroll
        for (int j = 0; j < 8; ++j) cnt += static_cast<int64_t>(v[j]) <= m0;
    }
    const int base = (cnt > 0 ? cnt - 1 : 0) << 4;
    int w[17];
#pragma unroll
    for (int j = 0; j < 17; ++j) w[j] = (base + j <= p.E) ? offs[base + j] : INT_MAX;
    int c2 = 0;
#pragma unroll
    for (int j = 0; j < 16; ++j) c2 += (base + j < p.E && static_cast<int64_t>(w[j]) <= m0);
    const int jj = c2 > 0 ? c2 - 1 : 0;
    const int lo = base + jj;
    int64_t e_begin = w[0], e_end = w[1];
#pragma unroll
    for (int j = 1; j < 16; ++j)
        if (j == jj) {
            e_begin = w[j];
            e_end = w[j + 1];
        }
    tl.run = mrows == 256 || (((m0 - e_begin) >> 7) & 1) == 0;
    tl.m_base = m0;
    tl.n0 = n0;
    tl.b_row0 = static_cast<int64_t>(lo) * p.b_rows + n0;
    tl.row_end = e_end;
    tl.expert = lo;
    return tl;
}

template <bool kGrouped, bool kSwiGLU, bool kShortWaits>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kPThreads, 1)
    nvfp4_gemm_pair_kernel(const __grid_constant__ CUtensorMap tma_a,
                           const __grid_constant__ CUtensorMap tma_b,
                           const __grid_constant__ CUtensorMap tma_y,
                           const __grid_constant__ CUtensorMap tma_sfa,
                           const __grid_constant__ CUtensorMap tma_sfb, GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    // the carve-up must fit behind the 1024-byte alignment (uniform in both CTAs)
    if (static_cast<size_t>(smem - smem_raw) + kPCarveBytes > kPSmemBytes) {
        if (threadIdx.x == 0) record_error(p.status, NVFP4_ERR_UNSUPPORTED_DEVICE, DETAIL_GEMM_DRAIN);
        return;
    }
    uint8_t* sA = smem;
    uint8_t* sB = sA + kPStages * kATileBytes;
    uint8_t* sSFA = sB + kPStages * kPBHalfBytes;
    uint8_t* sSFB = sSFA + kPStages * kSFATileBytes;
    uint8_t* sOut = sSFB + kPStages * kSFBTileBytes;              // 1024-aligned
    EpiInfo* info = reinterpret_cast<EpiInfo*>(sOut + kPOutBytes);
    int32_t* s_offsets = reinterpret_cast<int32_t*>(info + kInfoSlots);   // grouped: a copy of the offsets
    uint64_t* full = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(info) + kSBBytes);
    uint64_t* empty = full + kPStages;
    uint64_t* sf_ready = empty + kPStages;
    uint64_t* acc_full = sf_ready + kPStages;
    uint64_t* acc_empty = acc_full + 1;
    uint64_t* drain = acc_empty + 1;
    uint64_t* info_full = drain + 1;            // [kInfoSlots]
    uint64_t* info_empty = info_full + kInfoSlots;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(info_empty + kInfoSlots);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const bool leader = rank == 0;
    const int pair = blockIdx.x >> 1;
    const int npairs = gridDim.x >> 1;
    const int num_pm = static_cast<int>((p.M + 255) / 256);
    const int a_row_tiles = static_cast<int>((p.M + 127) / 128);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kPStages; ++s) {
            mbar_init(&full[s], 2);               // the A-side and the B-side producer
            mbar_init(&empty[s], 1);
            mbar_init(&sf_ready[s], 2 * kSFWarps);
        }
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, 2 * kEpiWarps);     // one arrival per epilogue warp of either CTA
        mbar_init(drain, 1);
        for (int s = 0; s < kInfoSlots; ++s) {
            mbar_init(&info_full[s], 1);          // the scheduler warp
            mbar_init(&info_empty[s], kEpiWarps);  // this CTA's epilogue warps
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        // collective across the pair: both CTAs get the same columns
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_u32(tmem_holder)), "r"(kTmemCols) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();     // both CTAs' barriers exist before any cross-CTA signal
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    pdl_wait();             // the producers of the operands and offsets have completed
    // Pipeline waits: the 2 s default, or the debug limit of the short-wait
    // instantiation (nvfp4_debug_set_gemm_wait_limit).
    auto wait_c = [&](uint64_t* bar, uint32_t parity) -> bool {
        return kShortWaits ? mbar_wait_cluster_short(bar, parity, p.wait_limit_ns, abort_flag)
                           : mbar_wait_cluster(bar, parity, kWaitLimitNs, abort_flag);
    };
    auto wait_b = [&](uint64_t* bar, uint32_t parity) -> bool {
        return kShortWaits ? mbar_wait_short(bar, parity, p.wait_limit_ns, abort_flag)
                           : mbar_wait_bounded(bar, parity, kWaitLimitNs, abort_flag);
    };
    int tiles = num_pm * p.num_n_tiles;
    int mrows = 128;   // grouped: rows per slot of the padded layout
    const int32_t* offs = p.offsets;   // grouped: where the expert lookups read the offsets
    int64_t used = p.M;   // grouped: rows of the layout in use (offsets[E])
    if (kGrouped) {
        // A layout whose expert segments are all 256-row aligned is walked in
        // 256-row slots, every one a pair tile (the strided assignment then
        // gives every pair the same number of tiles); otherwise in 128-row
        // slots, a pair tile starting at every second one of an expert.
        // the offsets, copied to shared memory when they fit beside the
        // tile-information ring: every role's expert lookups then cost
        // shared-memory latency instead of two rounds of L2 round trips
        bool misaligned = false;
        for (int e = threadIdx.x; e <= p.E; e += blockDim.x) {
            const int32_t o = __ldg(p.offsets + e);
            misaligned |= (o & 255) != 0;
            if (p.E + 1 <= kSmemOffsets) s_offsets[e] = o;
        }
        mrows = __syncthreads_or(misaligned) ? 128 : 256;
        if (p.E + 1 <= kSmemOffsets) offs = s_offsets;
        // slots of the padded layout in use: it ends at offsets[E]
        used = __ldg(p.offsets + p.E);
        if (used > p.M || used < 0) {
            if (threadIdx.x == 0) record_error(p.status, NVFP4_ERR_DEVICE_INPUT, DETAIL_EXPERT_OFFSETS);
            used = used < 0 ? 0 : p.M;
        }
        tiles = static_cast<int>((used + mrows - 1) / mrows) * p.num_n_tiles;
    }

    // Roles by warpgroup.  Each branch starts with its warpgroup's register
    // split (every warp of the warpgroup executes it, converged), so the code
    // of the branch is compiled within that register count.
    if (warp < kFirstSFWarp) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kSwiGLU ? kRegsWG0Swi : kRegsWG0));
        if ((warp == 0 || warp == kPBWarp) && lane < kPLoadLanes) {
            // ------------------------------ producers (both CTAs) ------------------
            // Warp 0 loads A and its scales, warp kPBWarp this CTA's 128 rows of B
            // and the B scales; kPLoadLanes lanes of each split the rows.  (One
            // lane per warp with 128-row boxes measured as fast as two or four
            // lanes with smaller boxes, and simpler.)  The scale atoms come by
            // tensor TMA too: with 2 KB non-tensor bulk copies the B producer,
            // which issues two of them per K step, fell ~1,000 cycles behind the
            // A producer and the K step took ~10% longer.
            const bool side_b = warp == kPBWarp;
            const int sub = lane;                     // which kPBoxRows-row part
            const CUtensorMap* map = side_b ? &tma_b : &tma_a;
            const CUtensorMap* sf_map = side_b ? &tma_sfb : &tma_sfa;
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(sf_map)) : "memory");
            uint32_t stage = 0, phase = 0;
            uint32_t issued_mask = 0, last_phase = 0;
            bool ok = true;
            for (int t = pair; t < tiles && ok; t += npairs) {
                const PairTile tl = pair_tile_at<kGrouped, kSwiGLU>(p, t, num_pm, mrows, offs);
                if (!tl.run) continue;
                if (kGrouped && !side_b && rank == 0 && (offs[tl.expert] & 127) != 0)
                    record_error(p.status, NVFP4_ERR_DEVICE_INPUT, DETAIL_EXPERT_OFFSETS);
                const int64_t m0 = tl.m_base + rank * 128;
                const int64_t n0 = tl.n0;
                const int a_tile = static_cast<int>(m0 / 128);
                const bool a_sf_ok = a_tile < a_row_tiles;
                // the B tile's two 128-row halves: consecutive rows, or (SwiGLU)
                // gate rows and the matching up rows; their scale atoms are one
                // box of the B scale map at 128-row tile nt128 (of the expert)
                const int nt128 = static_cast<int>(n0 / 128);
                const int64_t b_half1 = kSwiGLU ? p.ffn : 128;
                const int32_t sf_expert = kGrouped ? static_cast<int32_t>(tl.expert) : 0;
                for (int kt = 0; kt < p.num_k_tiles; ++kt) {
                    ok = __all_sync(kPLoadMask,
                                    wait_c(&empty[stage], phase ^ 1u));
                    if (!ok) break;
                    const int64_t g0 = static_cast<int64_t>(kt) * kMmaPerStage;
                    // lane 0 announces the side's bytes before any of its copies is
                    // issued (scale boxes are whole: past the last K group or the
                    // last tile they hold the zero fill, unused)
                    if (sub == 0)
                        mbar_arrive_expect_tx(&full[stage], side_b ? kPBHalfBytes + kSFBTileBytes
                                                                   : kATileBytes + (a_sf_ok ? kSFATileBytes : 0u));
                    __syncwarp(kPLoadMask);
                    if (!side_b) {
                        tma_load_2d(map, &full[stage], sA + stage * kATileBytes + sub * kPBoxRows * kBKBytes,
                                    kt * kBKBytes, static_cast<int32_t>(m0 + kPBoxRows * sub));
                        if (a_sf_ok && sub == 0)
                            tma_load_5d(sf_map, &full[stage], sSFA + stage * kSFATileBytes, 0,
                                        static_cast<int32_t>(2 * g0), a_tile, 0, 0);
                    } else {
                        tma_load_2d(map, &full[stage], sB + stage * kPBHalfBytes + sub * kPBoxRows * kBKBytes,
                                    kt * kBKBytes,
                                    static_cast<int32_t>(tl.b_row0 + rank * b_half1 + kPBoxRows * sub));
                        if (sub == 0)
                            tma_load_5d(sf_map, &full[stage], sSFB + stage * kSFBTileBytes, 0,
                                        static_cast<int32_t>(2 * g0), nt128, 0, sf_expert);
                    }
                    issued_mask |= 1u << stage;
                    last_phase = (last_phase & ~(1u << stage)) | (phase << stage);
                    if (++stage == kPStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                *abort_flag = 1;
                if (sub == 0) record_error(p.status, NVFP4_ERR_TIMEOUT, DETAIL_GEMM_PRODUCER);
            }
            // every copy this thread issued must land before the CTA may exit
            for (int s = 0; s < kPStages; ++s)
                if (issued_mask & (1u << s))
                    if (!mbar_wait_bounded(&full[s], (last_phase >> s) & 1u, kDrainLimitNs, nullptr))
                        record_error(p.status, NVFP4_ERR_TIMEOUT, DETAIL_GEMM_DRAIN);
        } else if (warp == 1 && leader) {
            // ------------------------------ MMA issuer (even CTA) ------------------
            // The whole warp runs the loop (warp-uniform control flow and
            // descriptors); one elected lane issues the MMAs and commits.
            uint32_t stage = 0, phase = 0, acc_phase = 0;
            bool ok = true;
            const uint64_t a_desc0 = sw128_desc(sA);
            const uint64_t b_desc0 = sw128_desc(sB);
            for (int t = pair; t < tiles && ok; t += npairs) {
                if (mrows != 256 && !pair_tile_at<kGrouped, kSwiGLU>(p, t, num_pm, mrows, offs).run) continue;
                ok = __all_sync(0xFFFFFFFFu, wait_c(acc_empty, acc_phase ^ 1u));
                if (!ok) break;
                tc_fence_after();
                for (int kt = 0; kt < p.num_k_tiles; ++kt) {
                    // both CTAs' scale warps have seen their stage full and written TMEM
                    ok = __all_sync(0xFFFFFFFFu,
                                    wait_c(&sf_ready[stage], phase));
                    if (!ok) break;
                    tc_fence_after();
                    const int ng = min(kMmaPerStage, p.kgroups - kt * kMmaPerStage);
                    const uint32_t sf_col = tmem + kSFTmemCol + stage * kSFTmemPerStage;
                    // descriptor start addresses advance in 16-byte units: 32 bytes per K step
                    const uint64_t ad = a_desc0 + stage * (kATileBytes >> 4);
                    const uint64_t bd = b_desc0 + stage * (kPBHalfBytes >> 4);
                    if (elect_one()) {
                        if (ng == kMmaPerStage) {
    #pragma unroll
                            for (int j = 0; j < kMmaPerStage; ++j)
                                tc_mma_pair(tmem, ad + 2 * j, bd + 2 * j, (kt > 0 || j > 0) ? 1u : 0u,
                                            sf_col + j * 4, sf_col + 16 + j * 8);
                        } else {
                            for (int j = 0; j < ng; ++j)
                                tc_mma_pair(tmem, ad + 2 * j, bd + 2 * j, (kt > 0 || j > 0) ? 1u : 0u,
                                            sf_col + j * 4, sf_col + 16 + j * 8);
                        }
                        tc_commit_pair_both(&empty[stage]);
                    }
                    __syncwarp();
                    if (++stage == kPStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                if (elect_one()) tc_commit_pair_both(acc_full);
                __syncwarp();
                acc_phase ^= 1u;
            }
            if (!ok) {
                *abort_flag = 1;
                if (lane == 0) record_error(p.status, NVFP4_ERR_TIMEOUT, DETAIL_GEMM_MMA);
            }
            // all tensor-core work issued by this warp completes before TMEM is freed
            if (elect_one()) tc_commit_pair(drain);
            __syncwarp();
            if (!mbar_wait_bounded(drain, 0u, kDrainLimitNs, nullptr) && lane == 0)
                record_error(p.status, NVFP4_ERR_TIMEOUT, DETAIL_GEMM_DRAIN);
        } else if (kGrouped && warp == kSchedWarp) {
            // ------------------------------ tile scheduler (both CTAs) -------------
            // For each tile of this pair, in order: the tile lookup (for grouped
            // layouts an expert search over the offsets, each load an L2 round
            // trip) and the loads of the tile's S_a rows and S_b columns, written
            // to the epilogue's ring one tile ahead, so that none of these
            // latencies sits between two tiles of the epilogue.
            uint32_t slot = 0, phase = 0;
            bool ok = true;
            for (int t = pair; t < tiles && ok; t += npairs) {
                const PairTile tl = pair_tile_at<kGrouped, kSwiGLU>(p, t, num_pm, mrows, offs);
                if (!tl.run) continue;
                const int64_t mrow0 = tl.m_base + rank * 128;
                float a[128 / 32], b[kBN / 32];
    #pragma unroll
                for (int i = 0; i < 128 / 32; ++i) {
                    const int64_t m = mrow0 + i * 32 + lane;
                    a[i] = (m < p.M) ? __ldg(p.sa + m * p.sa_stride) : 0.0f;
                }
                // the tile's 256 B rows: consecutive, or (SwiGLU) 128 gate rows
                // then the 128 matching up rows
                const float* sbp =
                    p.sb + p.sb_stride * ((kGrouped ? static_cast<int64_t>(tl.expert) * p.b_rows : 0) + tl.n0);
    #pragma unroll
                for (int i = 0; i < kBN / 32; ++i) {
                    const int c = i * 32 + lane;
                    if (kSwiGLU) {
                        b[i] = __ldg(sbp + (c < 128 ? c : p.ffn + c - 128) * p.sb_stride);
                    } else {
                        const int64_t n = tl.n0 + c;
                        b[i] = (n < p.N) ? __ldg(sbp + c * p.sb_stride) : 0.0f;
                    }
                }
                ok = __all_sync(0xFFFFFFFFu, wait_b(&info_empty[slot], phase ^ 1u));
                if (!ok) break;
                EpiInfo* e = info + slot;
    #pragma unroll
                for (int i = 0; i < 128 / 32; ++i) e->sa[i * 32 + lane] = a[i];
    #pragma unroll
                for (int i = 0; i < kBN / 32; ++i) e->sb[i * 32 + lane] = b[i];
                if (lane == 0) {
                    e->m_base = tl.m_base;
                    e->n0 = tl.n0;
                    // this CTA's 128 rows lie inside the tile's row range, or wholly past it
                    e->write = mrow0 < tl.row_end;
                    e->end = 0;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&info_full[slot]);
                if (++slot == kInfoSlots) {
                    slot = 0;
                    phase ^= 1u;
                }
            }
            if (ok) {
                // the end marker, once its slot is free
                ok = __all_sync(0xFFFFFFFFu, wait_b(&info_empty[slot], phase ^ 1u));
                if (ok && lane == 0) {
                    info[slot].end = 1;
                    mbar_arrive(&info_full[slot]);
                }
            }
            if (!ok) {
                *abort_flag = 1;
                if (lane == 0) record_error(p.status, NVFP4_ERR_TIMEOUT, DETAIL_GEMM_EPILOGUE);
            }
        }
    } else if (warp < kFirstEpiWarp) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kSwiGLU ? kRegsWG1Swi : kRegsWG1));
            // ------------------------------ scale warps (both CTAs) ----------------
            const int quad = warp & 3;
            const uint32_t t_lane = static_cast<uint32_t>(quad * 32) << 16;
            uint32_t stage = 0, phase = 0;
            bool ok = true;
            for (int t = pair; t < tiles && ok; t += npairs) {
                if (mrows != 256 && !pair_tile_at<kGrouped, kSwiGLU>(p, t, num_pm, mrows, offs).run) continue;
                for (int kt = 0; kt < p.num_k_tiles; ++kt) {
                    bool got = wait_b(&full[stage], phase);
                    got = __all_sync(0xFFFFFFFFu, got);
                    if (!got) {
                        ok = false;
                        break;
                    }
                    const int ng = min(kMmaPerStage, p.kgroups - kt * kMmaPerStage);
                    const uint4* sfa_s = reinterpret_cast<const uint4*>(sSFA + stage * kSFATileBytes);
                    const uint4* sfb_s = reinterpret_cast<const uint4*>(sSFB + stage * kSFBTileBytes);
                    uint32_t va[16], vb[32];
    #pragma unroll
                    for (int j = 0; j < kMmaPerStage; ++j) {
                        const uint4 a = (j < ng) ? sfa_s[j * 32 + lane] : make_uint4(0u, 0u, 0u, 0u);
                        const uint4 b0 = (j < ng) ? sfb_s[j * 32 + lane] : make_uint4(0u, 0u, 0u, 0u);
                        const uint4 b1 = (j < ng) ? sfb_s[(kSFATileBytes / 16) + j * 32 + lane]
                                                  : make_uint4(0u, 0u, 0u, 0u);
                        va[4 * j] = a.x; va[4 * j + 1] = a.y; va[4 * j + 2] = a.z; va[4 * j + 3] = a.w;
                        vb[8 * j] = b0.x; vb[8 * j + 1] = b0.y; vb[8 * j + 2] = b0.z; vb[8 * j + 3] = b0.w;
                        vb[8 * j + 4] = b1.x; vb[8 * j + 5] = b1.y; vb[8 * j + 6] = b1.z;
                        vb[8 * j + 7] = b1.w;
                    }
                    const uint32_t sf_col = tmem + t_lane + kSFTmemCol + stage * kSFTmemPerStage;
                    tmem_st16(sf_col, va);
                    tmem_st32(sf_col + 16, vb);
                    tmem_st_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster(peer_addr(&sf_ready[stage], 0));
                    if (++stage == kPStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                *abort_flag = 1;
                if (lane == 0) record_error(p.status, NVFP4_ERR_TIMEOUT, DETAIL_GEMM_MMA);
            }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kSwiGLU ? kRegsEpiSwi : kRegsEpi));
            // ------------------------------ epilogue (both CTAs) -------------------
            // Warp (quad, half) owns TMEM lanes quad*32.. and accumulator columns
            // half*128..: two rounds of 64 columns, each loaded with two tcgen05.ld
            // and one wait, scaled by S_a[m] S_b[n], rounded to bf16, written into
            // this warp's swizzled 32 x 64 staging box and stored by TMA (which
            // clips rows >= M and columns >= N).  With the SwiGLU epilogue the
            // warp instead loads gate columns half*64.. and the matching up
            // columns 128 + half*64.., rounds both to bf16 as the plain epilogue
            // would, and stores the 64 columns h = bf16(silu(g) u) of one box.
            const int quad = warp & 3;
            const int ew = warp - kFirstEpiWarp;
            const int half = ew >> 2;
            const uint32_t t_lanes = tmem + (static_cast<uint32_t>(quad * 32) << 16);
            // accumulator columns of the four 32-column loads
            const uint32_t c_first = kSwiGLU ? half * 64 : half * (kBN / 2);
            const uint32_t c_second = kSwiGLU ? 128 + half * 64 : half * (kBN / 2) + 64;
            uint8_t* box = sOut + ew * kPOutBoxBytes;
            uint8_t* my_row = box + lane * 128;
            const uint32_t acc_empty_leader = peer_addr(acc_empty, 0);
            float* sb_w = reinterpret_cast<float*>(info) + ew * (kBN / 2);   // dense: this warp's S_b half
            uint32_t acc_phase = 0, islot = 0, iphase = 0;
            int t = pair;
            for (;;) {
                bool write;
                int64_t row0, n_half;
                float sa;
                const float* sb_s;
                if constexpr (kGrouped) {
                    // the next tile's origin and scales, from the scheduler warp
                    bool got = wait_b(&info_full[islot], iphase);
                    got = __all_sync(0xFFFFFFFFu, got);
                    if (!got) {
                        *abort_flag = 1;
                        if (lane == 0) record_error(p.status, NVFP4_ERR_TIMEOUT, DETAIL_GEMM_EPILOGUE);
                        break;
                    }
                    const EpiInfo* ti = info + islot;
                    if (ti->end) break;
                    write = ti->write != 0;
                    row0 = ti->m_base + rank * 128 + quad * 32;
                    sa = ti->sa[quad * 32 + lane];
                    n_half = ti->n0 + half * (kSwiGLU ? 64 : kBN / 2);
                    sb_s = ti->sb + half * (kSwiGLU ? 64 : kBN / 2);
                } else {
                    if (t >= tiles) break;
                    const PairTile tl = pair_tile_at<false, false>(p, t, num_pm, mrows);
                    t += npairs;
                    // this CTA's 128 rows lie inside the tile's row range, or wholly past it
                    write = tl.m_base + rank * 128 < tl.row_end;
                    row0 = tl.m_base + rank * 128 + quad * 32;
                    const int64_t m = row0 + lane;
                    sa = (m < p.M) ? __ldg(p.sa + m * p.sa_stride) : 0.0f;
                    n_half = tl.n0 + half * (kBN / 2);
                    const float* sbp = p.sb + p.sb_stride * n_half;
                    __syncwarp();
    #pragma unroll
                    for (int i = 0; i < kBN / 2 / 32; ++i) {
                        const int64_t n = n_half + i * 32 + lane;
                        sb_w[i * 32 + lane] = (n < p.N) ? __ldg(sbp + (i * 32 + lane) * p.sb_stride) : 0.0f;
                    }
                    __syncwarp();
                    sb_s = sb_w;
                }
                bool ok = wait_c(acc_full, acc_phase);
                ok = __all_sync(0xFFFFFFFFu, ok);
                if (!ok) {
                    *abort_flag = 1;
                    if (lane == 0) record_error(p.status, NVFP4_ERR_TIMEOUT, DETAIL_GEMM_EPILOGUE);
                    break;
                }
                tc_fence_after();
                // Staging of 64 packed columns (one round): wait until the previous
                // store from this warp's box has read it, write the rows, then
                // (separately) fence and store the box with TMA.
                auto stage = [&](const uint32_t (&q)[16], const uint32_t (&q2)[16]) {
                    if (lane == 0) bulk_wait_read();
                    __syncwarp();
                    // 16-byte chunk j of row `lane` goes to chunk j ^ (lane % 8) (128-byte swizzle)
    #pragma unroll
                    for (int j = 0; j < 4; ++j)
                        *reinterpret_cast<uint4*>(my_row + ((j ^ (lane & 7)) << 4)) =
                            make_uint4(q[4 * j], q[4 * j + 1], q[4 * j + 2], q[4 * j + 3]);
    #pragma unroll
                    for (int j = 0; j < 4; ++j)
                        *reinterpret_cast<uint4*>(my_row + (((j + 4) ^ (lane & 7)) << 4)) =
                            make_uint4(q2[4 * j], q2[4 * j + 1], q2[4 * j + 2], q2[4 * j + 3]);
                };
                auto store = [&](int64_t x) {
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0 && write && row0 < p.M && x < p.N) {
                        tma_store_2d(&tma_y, box, static_cast<int32_t>(x), static_cast<int32_t>(row0));
                        bulk_commit();
                    }
                };
                // The warp's 128 accumulator columns are loaded in one round and the
                // accumulator released at once; scaling, staging and the stores
                // (two 64-column boxes) follow while the next tile's MMAs run.
                uint32_t r0[32], r1[32], r2[32], r3[32];
                tmem_ld32(t_lanes + c_first, r0);
                tmem_ld32(t_lanes + c_first + 32, r1);
                tmem_ld32(t_lanes + c_second, r2);
                tmem_ld32(t_lanes + c_second + 32, r3);
                tmem_wait(r0);
                reg_fence(r1);
                reg_fence(r2);
                reg_fence(r3);
                // every accumulator read of this tile is complete
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(acc_empty_leader);
                if constexpr (kGrouped && kSwiGLU) {
                    // g and u as the plain epilogue rounds them, then h = bf16(silu(g) u)
                    uint32_t qa[16], qb[16];
                    {
                        uint32_t qg[16], qu[16];
                        scale_chunk(r0, sb_s, sa, qg);
                        scale_chunk(r2, sb_s + 128, sa, qu);
    #pragma unroll
                        for (int j = 0; j < 16; ++j) qa[j] = swiglu_pair(qg[j], qu[j]);
                    }
                    {
                        uint32_t qg[16], qu[16];
                        scale_chunk(r1, sb_s + 32, sa, qg);
                        scale_chunk(r3, sb_s + 160, sa, qu);
    #pragma unroll
                        for (int j = 0; j < 16; ++j) qb[j] = swiglu_pair(qg[j], qu[j]);
                    }
                    // every read of this tile's ring slot is done
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&info_empty[islot]);
                    stage(qa, qb);
                    store(n_half);
                } else {
                {
                    uint32_t qa[16], qb[16];
                    scale_chunk(r0, sb_s, sa, qa);
                    scale_chunk(r1, sb_s + 32, sa, qb);
                    stage(qa, qb);
                    store(n_half);
                }
                {
                    uint32_t qa[16], qb[16];
                    scale_chunk(r2, sb_s + 64, sa, qa);
                    scale_chunk(r3, sb_s + 96, sa, qb);
                    if constexpr (kGrouped) {
                        // every read of this tile's ring slot is done
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&info_empty[islot]);
                    }
                    stage(qa, qb);
                    store(n_half + 64);
                }
                }
                acc_phase ^= 1u;
                if (kGrouped && ++islot == kInfoSlots) {
                    islot = 0;
                    iphase ^= 1u;
                }
            }
            // SwiGLU: the rows of H past the layout's used rows (no tile covers
            // them) are written as zeros, each CTA a slice, 16 bytes per lane
            if (kGrouped && kSwiGLU && used < p.M) {
                const int64_t tail = p.M - used;
                const int64_t per = (tail + gridDim.x - 1) / gridDim.x;
                const int64_t r_begin = used + static_cast<int64_t>(blockIdx.x) * per;
                const int64_t r_end = r_begin + per < p.M ? r_begin + per : p.M;
                const int pieces = static_cast<int>(p.ffn / 8);
                for (int64_t r = r_begin + ew; r < r_end; r += kEpiWarps)
                    for (int c = lane; c < pieces; c += 32)
                        reinterpret_cast<uint4*>(p.y + r * p.ld_y)[c] = make_uint4(0u, 0u, 0u, 0u);
            }
            // the staging boxes stay valid until the stores have finished
            if (lane == 0) bulk_wait_all();
            __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync_all();     // the pair's MMAs are done with both CTAs' SMEM and TMEM
    tc_fence_after();
    if (warp == 1) {
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmemCols) : "memory");
    }
}

// ----------------------------------------------------------------------------
// Host side
// ----------------------------------------------------------------------------
using EncodeTiledFn = TensorMapEncodeTiledFn;
EncodeTiledFn encode_fn() { return tensor_map_encode_fn(); }

// Rows of `row_bytes` packed bytes; box = 128 bytes x box_rows, 128-byte swizzle.
bool make_map(CUtensorMap* map, const void* base, int64_t rows, int64_t row_bytes, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(row_bytes), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_bytes)};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(kBKBytes), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A swizzled scale array (kgroups K groups per 128-row tile, 512-byte atoms)
// as [experts][halves][tiles][2 kgroups][256 bytes]; box = 8 rows (the four
// atoms of one K step) of box_tiles x box_halves tiles, no swizzle.  Boxes that
// reach past a dimension are zero-filled.
bool make_map_sf(CUtensorMap* map, const void* base, int64_t kgroups, int64_t tiles, int64_t halves,
                 int64_t experts, uint32_t box_tiles, uint32_t box_halves) {
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr || kgroups <= 0 || tiles <= 0 || halves <= 0 || experts <= 0) return false;
    if (tiles > INT32_MAX || experts > INT32_MAX || 2 * kgroups > INT32_MAX) return false;
    const cuuint64_t tile_bytes = static_cast<cuuint64_t>(kgroups) * kSFAtomBytes;
    cuuint64_t dims[5] = {kSFMapRowBytes, static_cast<cuuint64_t>(2 * kgroups), static_cast<cuuint64_t>(tiles),
                          static_cast<cuuint64_t>(halves), static_cast<cuuint64_t>(experts)};
    cuuint64_t strides[4] = {kSFMapRowBytes, tile_bytes, tile_bytes * tiles, tile_bytes * tiles * halves};
    cuuint32_t box[5] = {kSFMapRowBytes, kSFMapBoxRows, box_tiles, box_halves, 1};
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 5, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Y [rows x cols] bf16 with row pitch ld elements; box = 64 columns x 32 rows, 128-byte swizzle.
bool make_map_y(CUtensorMap* map, void* base, int64_t rows, int64_t cols, int64_t ld) {
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
    cuuint32_t box[2] = {64, 32};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool kGrouped, bool kSwiGLU, bool kShortWaits>
nvfp4_status launch_gemm_pair(const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& my,
                              const CUtensorMap& msfa, const CUtensorMap& msfb, const GemmParams& p, int64_t pair_tiles, const DeviceCtx& ctx, cudaStream_t s) {
    static unsigned long long attr_set[64] = {};   // per context: see ctx_cached
    if (!ctx_cached(attr_set, ctx)) {
        if (cudaFuncSetAttribute(nvfp4_gemm_pair_kernel<kGrouped, kSwiGLU, kShortWaits>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kPSmemBytes)) != cudaSuccess)
            return NVFP4_ERR_CUDA;
        ctx_cache_set(attr_set, ctx);
    }
    // persistent: as many pairs as can be resident at once (an SM left alone in
    // its GPC cannot host half of a pair)
    static int resident[64] = {};
    if (resident[ctx.device & 63] == 0) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(ctx.sm_count & ~1), 1, 1);
        cfg.blockDim = dim3(kPThreads, 1, 1);
        cfg.dynamicSmemBytes = kPSmemBytes;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, nvfp4_gemm_pair_kernel<kGrouped, kSwiGLU, kShortWaits>, &cfg) != cudaSuccess || n <= 0) {
            (void)cudaGetLastError();
            n = ctx.sm_count / 2;
        }
        resident[ctx.device & 63] = n;
    }
    const int64_t cap = resident[ctx.device & 63];
    const int64_t pairs = pair_tiles < cap ? pair_tiles : cap;
    if (pairs <= 0) return NVFP4_OK;
    // programmatic serialization: set-up (barriers, TMEM, tensor maps) overlaps
    // the producer kernel's tail; the kernel waits before reading its inputs
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs), 1, 1);
    cfg.blockDim = dim3(kPThreads, 1, 1);
    cfg.dynamicSmemBytes = kPSmemBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, nvfp4_gemm_pair_kernel<kGrouped, kSwiGLU, kShortWaits>, ma, mb, my, msfa, msfb, p) !=
        cudaSuccess)
        return NVFP4_ERR_CUDA;
    return NVFP4_OK;
}

// Pipeline wait limit of the next GEMM launches: the default, or a short limit
// set through nvfp4_debug_set_gemm_wait_limit to exercise the abort path.
std::atomic<uint64_t> g_wait_limit_ns{kWaitLimitNs};

nvfp4_status check_operand_shapes(int64_t N, int64_t K) {
    if (N <= 0 || N % 16 != 0 || K <= 0 || K % 64 != 0) return NVFP4_ERR_SHAPE;
    if (K > (int64_t(1) << 20) || N > (int64_t(1) << 24)) return NVFP4_ERR_SHAPE;
    return NVFP4_OK;
}

}  // namespace
}  // namespace nvfp4

using namespace nvfp4;

extern "C" {

nvfp4_status nvfp4_gemm_ex(const void* a_q, const void* a_sf, const float* a_s, int32_t a_s_per_row,
                           int64_t M, const void* b_q, const void* b_sf, const float* b_s,
                           int32_t b_s_per_row, int64_t N, int64_t K, void* y, int64_t ld_y,
                           nvfp4_stream_t stream) {
    DeviceCtx ctx;
    nvfp4_status st = device_ctx(&ctx);
    if (st != NVFP4_OK) return st;
    if (M < 0 || M > (int64_t(1) << 31) - kBM) return NVFP4_ERR_SHAPE;
    if ((st = check_operand_shapes(N, K)) != NVFP4_OK) return st;
    if (ld_y < N || ld_y % 8 != 0) return NVFP4_ERR_SHAPE;
    if (M == 0) return NVFP4_OK;
    if (!a_q || !a_sf || !a_s || !b_q || !b_sf || !b_s || !y) return NVFP4_ERR_INVALID_ARG;
    if (!aligned(a_q, 16) || !aligned(b_q, 16) || !aligned(a_sf, 16) || !aligned(b_sf, 16) ||
        !aligned(y, 16) || !aligned(a_s, 4) || !aligned(b_s, 4))
        return NVFP4_ERR_ALIGNMENT;
    CUtensorMap ma, mb, my, msfa, msfb;
    // pairs of CTAs: each loads a 128-row half of the 256-row B tile
    if (!make_map(&ma, a_q, M, K / 2, kPBoxRows) || !make_map(&mb, b_q, N, K / 2, kPBoxRows) ||
        !make_map_y(&my, y, M, N, ld_y) ||
        !make_map_sf(&msfa, a_sf, K / 64, ceil_div(M, 128), 1, 1, 1, 1) ||
        !make_map_sf(&msfb, b_sf, K / 64, ceil_div(N, 128), 1, 1, 2, 1))
        return NVFP4_ERR_CUDA;
    GemmParams p;
    p.sfa = static_cast<const uint8_t*>(a_sf);
    p.sfb = static_cast<const uint8_t*>(b_sf);
    p.sa = a_s;
    p.sb = b_s;
    p.y = static_cast<uint16_t*>(y);
    p.offsets = nullptr;
    p.status = ctx.status;
    p.M = M;
    p.N = N;
    p.ld_y = ld_y;
    p.sfb_expert_bytes = 0;
    p.kgroups = static_cast<int>(K / 64);
    p.num_k_tiles = static_cast<int>(ceil_div(K, 256));
    p.num_n_tiles = static_cast<int>(ceil_div(N, kBN));
    p.num_m_tiles = static_cast<int>(ceil_div(M, kBM));
    p.E = 0;
    p.sa_stride = a_s_per_row ? 1 : 0;
    p.sb_stride = b_s_per_row ? 1 : 0;
    p.n_fast = N < M ? 1 : 0;
    p.wait_limit_ns = g_wait_limit_ns.load();
    p.swiglu = 0;
    p.ffn = 0;
    p.b_rows = N;
    p.n_step = kBN;
    const int64_t pair_tiles = ceil_div(M, 256) * p.num_n_tiles;
    if (pair_tiles > (int64_t(1) << 30)) return NVFP4_ERR_SHAPE;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    return p.wait_limit_ns == kWaitLimitNs
               ? launch_gemm_pair<false, false, false>(ma, mb, my, msfa, msfb, p, pair_tiles, ctx, s)
               : launch_gemm_pair<false, false, true>(ma, mb, my, msfa, msfb, p, pair_tiles, ctx, s);
}

nvfp4_status nvfp4_gemm(const void* a_q, const void* a_sf, const float* a_s, int64_t M,
                        const void* b_q, const void* b_sf, const float* b_s, int64_t N, int64_t K,
                        void* y, int64_t ld_y, nvfp4_stream_t stream) {
    return nvfp4_gemm_ex(a_q, a_sf, a_s, 1, M, b_q, b_sf, b_s, 1, N, K, y, ld_y, stream);
}

}  // extern "C"

namespace nvfp4 {
namespace {

// The grouped GEMM, plain (Y [rows, N]) or with the SwiGLU epilogue
// (H [rows, F], N = F, B rows per expert 2F).
nvfp4_status grouped_gemm(const void* a_q, const void* a_sf, const float* a_s, int64_t rows_capacity,
                          const int32_t* expert_offsets, int32_t E, const void* b_q, const void* b_sf,
                          const float* b_s, int64_t N, int64_t K, void* y, bool swiglu, cudaStream_t stream) {
    DeviceCtx ctx;
    nvfp4_status st = device_ctx(&ctx);
    if (st != NVFP4_OK) return st;
    if (rows_capacity < 0 || rows_capacity > (int64_t(1) << 31) - kBM) return NVFP4_ERR_SHAPE;
    if (E < 1 || E > 1024) return NVFP4_ERR_SHAPE;
    const int64_t b_rows = swiglu ? 2 * N : N;
    if ((st = check_operand_shapes(b_rows, K)) != NVFP4_OK) return st;
    if (swiglu && N % 128 != 0) return NVFP4_ERR_SHAPE;
    if (rows_capacity == 0) return NVFP4_OK;
    if (!a_q || !a_sf || !a_s || !expert_offsets || !b_q || !b_sf || !b_s || !y)
        return NVFP4_ERR_INVALID_ARG;
    if (!aligned(a_q, 16) || !aligned(b_q, 16) || !aligned(a_sf, 16) || !aligned(b_sf, 16) ||
        !aligned(y, 16) || !aligned(a_s, 4) || !aligned(b_s, 4) || !aligned(expert_offsets, 4))
        return NVFP4_ERR_ALIGNMENT;
    CUtensorMap ma, mb, my, msfa, msfb;
    if (!make_map(&ma, a_q, rows_capacity, K / 2, kPBoxRows) ||
        !make_map(&mb, b_q, static_cast<int64_t>(E) * b_rows, K / 2, kPBoxRows) ||
        !make_map_y(&my, y, rows_capacity, N, N) ||
        !make_map_sf(&msfa, a_sf, K / 64, ceil_div(rows_capacity, 128), 1, 1, 1, 1) ||
        !(swiglu ? make_map_sf(&msfb, b_sf, K / 64, N / 128, 2, E, 1, 2)
                 : make_map_sf(&msfb, b_sf, K / 64, ceil_div(b_rows, 128), 1, E, 2, 1)))
        return NVFP4_ERR_CUDA;
    GemmParams p;
    p.sfa = static_cast<const uint8_t*>(a_sf);
    p.sfb = static_cast<const uint8_t*>(b_sf);
    p.sa = a_s;
    p.sb = b_s;
    p.y = static_cast<uint16_t*>(y);
    p.offsets = expert_offsets;
    p.status = ctx.status;
    p.M = rows_capacity;
    p.N = N;
    p.ld_y = N;
    p.sfb_expert_bytes = static_cast<int64_t>(nvfp4_sf_bytes(b_rows, K));
    p.kgroups = static_cast<int>(K / 64);
    p.num_k_tiles = static_cast<int>(ceil_div(K, 256));
    p.n_step = swiglu ? 128 : kBN;
    p.num_n_tiles = static_cast<int>(ceil_div(N, p.n_step));
    p.num_m_tiles = static_cast<int>(ceil_div(rows_capacity, kBM));
    p.E = E;
    p.sa_stride = 1;
    p.sb_stride = 1;
    p.n_fast = 0;
    p.wait_limit_ns = g_wait_limit_ns.load();
    p.swiglu = swiglu ? 1 : 0;
    p.ffn = swiglu ? N : 0;
    p.b_rows = b_rows;
    // slots: every 128-row tile of the capacity x every n-tile (about half start a pair tile)
    const int64_t slots = static_cast<int64_t>(p.num_m_tiles) * p.num_n_tiles;
    if (slots > (int64_t(1) << 31) - 1) return NVFP4_ERR_SHAPE;
    const int64_t pair_tiles = (slots + 1) / 2;
    if (p.wait_limit_ns != kWaitLimitNs)   // debug: short pipeline waits (not for the SwiGLU epilogue)
        return swiglu ? NVFP4_ERR_INVALID_ARG : launch_gemm_pair<true, false, true>(ma, mb, my, msfa, msfb, p, pair_tiles, ctx, stream);
    return swiglu ? launch_gemm_pair<true, true, false>(ma, mb, my, msfa, msfb, p, pair_tiles, ctx, stream)
                  : launch_gemm_pair<true, false, false>(ma, mb, my, msfa, msfb, p, pair_tiles, ctx, stream);
}

}  // namespace
}  // namespace nvfp4

extern "C" {

nvfp4_status nvfp4_grouped_gemm(const void* a_q, const void* a_sf, const float* a_s,
                                int64_t rows_capacity, const int32_t* expert_offsets, int32_t E,
                                const void* b_q, const void* b_sf, const float* b_s, int64_t N,
                                int64_t K, void* y, nvfp4_stream_t stream) {
    return grouped_gemm(a_q, a_sf, a_s, rows_capacity, expert_offsets, E, b_q, b_sf, b_s, N, K, y, false,
                        reinterpret_cast<cudaStream_t>(stream));
}

nvfp4_status nvfp4_grouped_gemm_swiglu(const void* a_q, const void* a_sf, const float* a_s,
                                       int64_t rows_capacity, const int32_t* expert_offsets, int32_t E,
                                       const void* b_q, const void* b_sf, const float* b_s, int64_t ffn,
                                       int64_t K, void* h, nvfp4_stream_t stream) {
    return grouped_gemm(a_q, a_sf, a_s, rows_capacity, expert_offsets, E, b_q, b_sf, b_s, ffn, K, h, true,
                        reinterpret_cast<cudaStream_t>(stream));
}

nvfp4_status nvfp4_debug_set_gemm_wait_limit(int64_t limit_ns) {
    if (limit_ns < 0 || limit_ns > 10000000000LL) return NVFP4_ERR_INVALID_ARG;
    g_wait_limit_ns.store(limit_ns == 0 ? kWaitLimitNs : static_cast<uint64_t>(limit_ns));
    return NVFP4_OK;
}

}  // extern "C"
