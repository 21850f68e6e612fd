// Grouped MXFP4 expert GEMMs on the 5th-generation tensor cores (tcgen05):
//   gate/up + SwiGLU   h = silu(x W_gate^T) * (x W_up^T)
//   down               slot_tj = w_tj * (h_tj W_down^T), summed over j by the
//                      combine launch that follows
//
// Sources: "A 297-line kernel file that decodes faster than vLLM", section "Where
// the time went" (rows "MoE gate/up + SwiGLU" and "MoE down + combine") and
// section "Optimizations" (row "MXFP4 MoE on tensor cores": weights re-laid out
// once at load, one grouped kernel for any token count; row "MoE token tile
// follows tokens per expert").
//
// Design (swap-AB): the MMA's M dimension is 128 weight rows (output features), N
// covers the tile's token rows, K runs over the contraction 256 values (one 128-byte
// row segment) per pipeline stage.  A = the MXFP4 weights exactly as stored (packed
// E2M1 codes, TMA boxes with the 128-byte swizzle); B = the activations, encoded as
// four packed E2M1 terms with their own E8M0 block scales, one pre-swizzled bulk
// copy per stage.  kind::mxf4 consumes both codes and both scale sets natively
// (K = 64 per instruction, scales copied into tensor memory with tcgen05.cp).  For
// 16-row decode tiles the four terms are concatenated along N (one N = 64 MMA per K
// step and weight tile; the epilogue adds the four column groups); larger tiles run
// one MMA per term into the same accumulator.
//
// Persistent CTAs (one per SM) take whole work units (expert tile x M tile)
// round-robin.  Warp roles: warp 0 issues TMA loads into a ring of shared-memory
// stages, warps 1 and 6 issue MMAs into tensor-memory accumulators, warps 2-5 (and
// 7-10 for 128-token tiles) run the epilogue of one unit while the MMAs of the next
// proceed.
//
// The W16 instances run the same kernel on bf16 weights and activations
// ("triton-kernels" README, "Fused MoE Dispatch": the Mixtral-style layer):
// kind::f16 MMAs with K = 16, 64-value stages of the same 128-byte rows, no scales,
// weights prepared into swizzled 16 KB tiles (one bulk copy each), and bf16 h
// written by the gate/up epilogue.
#include <type_traits>

#include "moe_common.cuh"
#include "moe_kernels.cuh"
#include "sm100_ptx.cuh"

namespace moe {

using namespace ptx;

namespace {

// warps: 0 TMA producer, 1 MMA issuer, 2-5 epilogue (one per tensor-memory lane
// quarter), 6 second MMA issuer (used when a stage carries two weight tiles)
constexpr int kSecondIssuerWarp = 6;
constexpr uint64_t kWaitLimit = 1000000000ull;  // ns a bounded mbarrier wait may take (1 s)

// MPAIR (down only): two neighbouring 128-row M tiles per work unit, sharing each
// stage's B tile, so a stage carries twice the weight bytes per activation byte.
// W16: bf16 weights and activations (kind::f16, no scales, one term per token).
template <int BM, bool GATEUP, bool MPAIR, bool W16 = false>
struct GemmCfg {
  static constexpr int kA = (GATEUP || MPAIR) ? 2 : 1;       // weight tiles per stage (gate/up, or 2 M tiles)
  static constexpr int kKStage = W16 ? 64 : gemm_kstage(BM); // K values per stage
  static constexpr int kKBytes = W16 ? 128 : kKStage / 2;    // bytes per operand row per stage
  static constexpr int kAtoms = W16 ? 0 : kKStage / kKGroup; // scale atoms per 128 rows per stage
  static constexpr int kKSteps = W16 ? kKStage / 16 : kKStage / 64;  // MMA K steps (32 bytes of every row)
  static constexpr int kATileBytes = kMTile * kKBytes;       // one 128-row weight tile of a stage
  static constexpr int kRowTerms = W16 ? 1 : kTerms;         // B rows per token
  static constexpr bool kConcat = !W16 && kTerms * BM <= 64; // all terms in one MMA along N
  static constexpr int kN = kConcat ? kTerms * BM : BM;      // MMA N
  static constexpr int kAccN = kN;                           // accumulator columns per weight tile
  // Decode stages that carry one weight tile (the unpaired down GEMM, 16-row tiles):
  // the stage's two K groups go to two MMA-issuing threads, each with its own scale
  // copies and its own accumulator slice, and the epilogue adds the two slices.  One
  // thread then issues half the tcgen05 instructions of a stage; at these shapes the
  // issuing thread, not the tensor pipe or the copies, sets the stage rate.
  static constexpr bool kSplitK = !W16 && kA == 1 && kConcat;
  static constexpr int kAccSlices = kSplitK ? 2 : kA;       // accumulator slices per buffer
  static constexpr int kAccCols = kAccSlices * kAccN;
  static constexpr int kVals = kA * BM;                      // values per row after summing terms
  static constexpr int kBRows = kRowTerms * BM;              // B tile rows (terms x token rows)
  static constexpr int kBBytes = kBRows * kKBytes;
  static constexpr int kNbAtoms = W16 ? 0 : (kBRows + 127) / 128;  // B scale atoms per stage
  static constexpr int kSfBytes = (kA + kNbAtoms) * kAtoms * kSfAtomBytes;
  static constexpr int kStageRaw = kA * kATileBytes + kBBytes + kSfBytes;
  static constexpr int kStageBytes = (kStageRaw + 1023) / 1024 * 1024;
  // the epilogue reads the whole accumulator into registers before releasing it
  static constexpr bool kLoadAll = kAccCols <= 128;
  // larger tiles: two epilogue warp groups take alternate 16-column chunks of the
  // accumulator (its long encode of h is latency-bound with one warp per scheduler)
  static constexpr int kEpiGroups = kLoadAll ? 1 : 2;
  static constexpr int kThreads = 224 + 128 * (kEpiGroups - 1);
  static constexpr int kMetaRows = BM > 128 ? BM : 128;      // row metadata entries (down epilogue)
  static constexpr int kEpiGroupBytes = 16 * kMTile * 4 + 2 * kMetaRows * 4;  // h transpose chunk + row metadata
  static constexpr int kEpiBytes = kEpiGroups * kEpiGroupBytes;
  static constexpr int kBarBytes = 2048;
  // two groups: the whole 227 KB a block may have (two stages of the largest tile);
  // one group: the depth measured best for the small tiles (a fifth BM=16 stage was
  // slower).  The split-K decode down GEMM stops at six: it issues its weight stages
  // while gate/up still streams, and a seventh and eighth measured slower at batch 1.
  static constexpr int kSmemBudget =
      kEpiGroups == 2 ? 232448 - 1024 /*align*/ - kBarBytes - kEpiBytes : 216 * 1024 - kEpiBytes;
  static constexpr int kStagesRaw = kSmemBudget / kStageBytes;
  static constexpr int kMaxStages = kSplitK ? 6 : 12;
  static constexpr int kStages = kStagesRaw > kMaxStages ? kMaxStages : kStagesRaw;
  static constexpr int kSmemBytes = kStages * kStageBytes + 1024 /*align*/ + kBarBytes + kEpiBytes;
  static constexpr uint32_t kTxNoB = kA * kATileBytes + kSfBytes;                // all but the B codes
  // MMA issuers: with two weight tiles per stage each of two threads issues one
  // tile's MMAs (its own accumulator, scale copies and B scale columns); with split K
  // groups each issues one K group's (the B scale atoms are then not duplicated)
  static constexpr int kIssuers = kSplitK ? 2 : kA;
  static constexpr int kSfColsPerStage = 4 * (kA + (kSplitK ? 1 : kIssuers) * kNbAtoms) * kAtoms;
  static constexpr int kSfCols = kStages * kSfColsPerStage;
  static constexpr int kNumAcc = (2 * kAccCols + kSfCols <= 512) ? 2 : 1;
  static constexpr int kTmemNeed = kNumAcc * kAccCols + kSfCols;
  static constexpr int kTmemCols = kTmemNeed <= 32 ? 32 : kTmemNeed <= 64 ? 64 : kTmemNeed <= 128 ? 128
                                   : kTmemNeed <= 256 ? 256 : 512;
  static_assert(kTmemNeed <= 512, "tensor memory budget");
  static_assert(kStages >= 2, "pipeline depth");
};

// Raster: units are grouped in blocks of `group` tiles; within a block the M tile
// varies slowest, so neighbouring units share weight tiles (same expert) and
// activation tiles through L2.
__device__ __forceinline__ void map_unit(int u, int num_tiles, int mt_count, int group, int& tile, int& mt) {
  const int g = u / (group * mt_count);
  const int first = g * group;
  const int gsize = min(group, num_tiles - first);
  const int within = u - first * mt_count;
  mt = within / gsize;
  tile = first + within % gsize;
}

// Work schedule of one CTA: whole units dealt round-robin (unit c + i*G).  With no
// more units than CTAs every CTA runs one unit (grid = U).  No unit is ever split
// along K: measured on the decode shapes, exchanging fp32 partials between CTAs for
// the last wave costs more than the last wave's imbalance.
struct Schedule {
  int KG, G, c, nseg;
  __device__ void init(int U, int kg, int grid, int cta) {
    KG = kg;
    G = grid;
    c = cta;
    nseg = (U > cta) ? (U - cta + grid - 1) / grid : 0;  // units cta, cta + G, ... below U
  }
  // segment i: its unit and K-group range (always the whole K)
  __device__ void seg(int i, int& u, int& kk0, int& kk1, bool& whole) const {
    u = c + i * G;
    kk0 = 0;
    kk1 = KG;
    whole = true;
  }
};

// silu(g) = g / (1 + e^-g) with the fast exponential and division (|error| well below
// the E2M1 encoding error that follows)
__device__ __forceinline__ float silu_f(float g) { return __fdividef(g, 1.f + __expf(-g)); }



}  // namespace

template <int BM, bool GATEUP, bool MPAIR, bool W16>
__global__ void __launch_bounds__(GemmCfg<BM, GATEUP, MPAIR, W16>::kThreads, 1)
    moe_gemm_kernel(const __grid_constant__ GemmParams p) {
  using C = GemmCfg<BM, GATEUP, MPAIR, W16>;
  extern __shared__ uint8_t gemm_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(gemm_smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + C::kStages * C::kStageBytes);
  uint64_t* empty_bar = full_bar + C::kStages;
  uint64_t* accf_bar = empty_bar + C::kStages;   // [2] accumulator ready
  uint64_t* acce_bar = accf_bar + 2;             // [2] accumulator drained
  uint64_t* drain_bar = acce_bar + 2;            // every MMA issuer's tensor-core work has completed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain_bar + 1);
  int* s_flags = reinterpret_cast<int*>(tmem_slot + 4);  // [0] error, [1] unit finisher
  // per epilogue group: h transpose [16][128], row assignment [128], its top-k weight [128]
  uint8_t* epi_smem = smem + C::kStages * C::kStageBytes + C::kBarBytes;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // prologue that touches nothing the previous kernel writes: barriers, tensor
  // memory, descriptor prefetch; it overlaps the previous kernel's tail
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], C::kIssuers);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&accf_bar[b], C::kIssuers);
      mbar_init(&acce_bar[b], 128 * C::kEpiGroups);
    }
    mbar_init(drain_bar, C::kIssuers);
    s_flags[0] = 0;
    fence_mbar_init();
  }
  if constexpr (!W16) {  // bf16 weights come by bulk copy, with no tensor map
    if (warp == 0 && lane == 0) tma_prefetch_desc(&p.tm_w);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_launch_dependents();
  // The tile table was written by the routing launch, which has completed before
  // this kernel can start: at least one launch lies between them, and every such
  // launch signals its dependents only after its own dependency wait.  So the table
  // is read before this kernel's wait; the B operand (gathered x, or h) comes from
  // the immediately preceding kernel and is only touched after pdl_wait().  Routing
  // outputs are read through L2 only (ld.global.cg): kernels overlap their
  // neighbours, so nothing may come from an L1 line left by an earlier call.
  // With single-tile raster groups a CTA's first unit is (tile blockIdx / mt, M unit
  // blockIdx % mt) whatever the tile count, so its tile entry is loaded together with
  // the count instead of after it (one L2 round trip less before the first copy).
  const int first_tile = (int)blockIdx.x / p.mt;
  const bool first_known = p.group_tiles == 1 && first_tile < p.max_tiles;
  const int4 first_te = first_known ? __ldcg(reinterpret_cast<const int4*>(p.tiles + first_tile)) : make_int4(0, 0, 0, 0);
  const int num_tiles = __ldcg(p.num_tiles);
  const int KG = p.kg;
  const int U = num_tiles * p.mt;
  const int grid = U <= (int)gridDim.x ? U : (int)gridDim.x;
  Schedule sch;
  sch.init(U, KG, grid > 0 ? grid : 1, blockIdx.x);
  if (U == 0 || (int)blockIdx.x >= grid) sch.nseg = 0;  // no work: straight to teardown

  auto stage_ptr = [&](int s) { return smem + s * C::kStageBytes; };
  // stage layout: [A tiles][B tile (terms x rows)][SF A: kA x kAtoms atoms][SF B: kAtoms x kNbAtoms atoms]
  auto a_tile = [&](int s, int j) { return stage_ptr(s) + j * C::kATileBytes; };
  auto b_tile = [&](int s) { return stage_ptr(s) + C::kA * C::kATileBytes; };
  auto sf_a = [&](int s, int j) {
    return stage_ptr(s) + C::kA * C::kATileBytes + C::kBBytes + j * C::kAtoms * kSfAtomBytes;
  };
  auto sf_b = [&](int s) { return stage_ptr(s) + C::kA * C::kATileBytes + C::kBBytes + C::kA * C::kAtoms * kSfAtomBytes; };

  const int kblocks = p.K / kMxBlock;  // real MX blocks along K; K steps past them are skipped

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    // The whole warp runs the ring in step with identical values (uniform control
    // flow); lane 0 alone issues each copy, through a predicate.  After the dependency
    // wait the activation copies of the stages issued before it go out from one lane
    // each, in parallel.
    __shared__ int s_pre[3][C::kStages];  // pre-issued stages: tile, K group, B rows
    const bool leader = lane == 0;
    // iterator over this CTA's (segment, K group) iterations
    int si = 0, kk = 0, kk1 = 0, tile = 0, mt = 0, expert = 0, b_rows = C::kBRows;
    auto open_seg = [&]() {
      int u, kk0;
      bool whole;
      sch.seg(si, u, kk0, kk1, whole);
      kk = kk0;
      map_unit(u, num_tiles, p.mt, p.group_tiles, tile, mt);
      TileEntry te;
      if (si == 0 && first_known) {
        te.expert = first_te.x;
        te.n_rows = first_te.z;
      } else {
        te = load_tile(p.tiles + tile);
      }
      expert = te.expert;
      // token-major tiles: only the real tokens' rows (kTerms per token) are loaded
      // (the MMA's columns of rows never loaded are never read)
      b_rows = (C::kConcat || W16) ? C::kRowTerms * max(1, min(te.n_rows, BM)) : C::kBRows;
    };
    auto advance = [&]() {
      if (++kk == kk1 && ++si < sch.nseg) open_seg();
    };
    // bytes the stage's barrier expects for the current tile
    auto tx_bytes = [&]() -> uint32_t { return C::kTxNoB + (uint32_t)b_rows * (uint32_t)C::kKBytes; };
    // Weights are read once per call.  When more units than CTAs stream them, mark
    // them evict-first so that the activation tiles every unit of a tile re-reads
    // stay in L2; a single wave keeps the normal policy (faster there).
    const uint64_t w_policy = U > grid ? l2_policy_evict_first() : l2_policy_evict_normal();
    auto load_a = [&](int s) {
      for (int j = 0; j < C::kA; ++j) {
        // gate/up: group j of M tile mt; down: M tile mt (or 2 mt + j), group 0.  An M
        // tile past the matrix reads zeros (TMA fill) and scales of the last tile.
        const int mrow = GATEUP ? mt : (MPAIR ? 2 * mt + j : mt);
        const int grp = GATEUP ? j : 0;
        if constexpr (W16) {
          // bf16: the prepared 16 KB tile in one bulk copy (the zero tile after the
          // last one for an M tile past the matrix)
          static_assert(!W16 || C::kATileBytes == kW16TileBytes, "prepared bf16 tile");
          const size_t ntiles = (size_t)p.E * p.w_groups * p.w_mt * p.kg;
          const size_t ti =
              mrow < p.w_mt ? (((size_t)expert * p.w_groups + grp) * p.w_mt + mrow) * p.kg + kk : ntiles;
          bulk_load_hint_if(leader, a_tile(s, j), p.w_tiles + ti * kW16TileBytes, (uint32_t)kW16TileBytes,
                            &full_bar[s], w_policy);
          continue;
        }
        tma_load_3d_hint_if(leader, a_tile(s, j), &p.tm_w, &full_bar[s], kk * C::kKBytes, mrow * kMTile,
                            expert * p.w_groups + grp, w_policy);
        const int msf = min(mrow, p.w_mt - 1);
        const uint8_t* wsf =
            p.w_sf + (((size_t)expert * p.w_groups + grp) * p.w_mt + msf) * (size_t)p.kg_sf * kSfAtomBytes;
        bulk_load_hint_if(leader, sf_a(s, j), wsf + (size_t)kk * C::kAtoms * kSfAtomBytes, C::kAtoms * kSfAtomBytes,
                          &full_bar[s], w_policy);
      }
    };
    // the (stage, tile) image of the activations is contiguous and already swizzled:
    // one bulk copy, and one for the stage's adjacent K groups of scale atoms
    auto load_b = [&](bool issue, int s, int b_tile_idx, int b_kk, int rows) {
      bulk_load_if(issue, b_tile(s),
                   p.act_q + ((size_t)b_kk * p.max_tiles + b_tile_idx) * (size_t)(C::kBRows * C::kKBytes),
                   (uint32_t)rows * (uint32_t)C::kKBytes, &full_bar[s]);
      if constexpr (W16) return;
      bulk_load_if(issue, sf_b(s),
                   p.act_sf + ((size_t)b_tile_idx * p.kg_sf + (size_t)b_kk * C::kAtoms) * (kSfAtomBytes * C::kNbAtoms),
                   C::kAtoms * C::kNbAtoms * kSfAtomBytes, &full_bar[s]);
    };
    auto wait_warp = [](uint64_t* bar, uint32_t parity, uint64_t limit) {
      return __shfl_sync(0xffffffffu, mbar_wait_bounded(bar, parity, limit) ? 1 : 0, 0) != 0;
    };
    int npre = 0;
    if (sch.nseg > 0) {
      open_seg();
      // weights of the first stages depend only on the routing: stream them while
      // the previous kernel finishes
      while (npre < C::kStages && si < sch.nseg) {
        mbar_arrive_expect_tx_if(leader, &full_bar[npre], tx_bytes());  // fresh stages: no wait
        load_a(npre);
        if (leader) {
          s_pre[0][npre] = tile;
          s_pre[1][npre] = kk;
          s_pre[2][npre] = b_rows;
        }
        ++npre;
        advance();
      }
    }
    __syncwarp();  // s_pre written by lane 0 is visible to the warp
    pdl_wait();
    if (lane < npre) load_b(true, lane, s_pre[0][lane], s_pre[1][lane], s_pre[2][lane]);
    __syncwarp();
    int g = npre;
    for (; si < sch.nseg; ++g) {
      const int s = g % C::kStages;
      const uint32_t ph = (g / C::kStages) & 1;
      if (!wait_warp(&empty_bar[s], ph ^ 1, p.wait_ns)) {
        if (leader) report_status(p.status, kStatusTimeoutProducer);
        s_flags[0] = 1;
        break;
      }
      mbar_arrive_expect_tx_if(leader, &full_bar[s], tx_bytes());
      load_a(s);
      load_b(leader, s, tile, kk, b_rows);
      advance();
    }
    // Before the CTA exits and its shared memory is reused, every copy issued into it
    // has landed: wait (bounded by the long limit, whatever the call's wait limit) for
    // the last ring's worth of stages.  On the normal path they were consumed already.
    for (int gg = max(0, g - C::kStages); gg < g; ++gg)
      wait_warp(&full_bar[gg % C::kStages], (gg / C::kStages) & 1, kWaitLimit);
  } else if (warp == 1 || warp == kSecondIssuerWarp) {
    // ------------------------------------------------------------ MMA issuers
    pdl_wait();
    const int issuer = warp == 1 ? 0 : 1;
    if (issuer < C::kIssuers) {
      // The whole warp runs this loop in step with identical values (its control flow
      // is warp-uniform, so descriptors and addresses can live in uniform registers);
      // lane 0 alone issues each tcgen05 instruction, through a predicate.
      const bool leader = lane == 0;
      // this warp's weight tiles [j0, j1) and K steps [ks0, ks1) of every stage
      constexpr bool kTilePerIssuer = C::kIssuers == 2 && !C::kSplitK;
      const int j0 = kTilePerIssuer ? issuer : 0, j1 = kTilePerIssuer ? issuer + 1 : C::kA;
      const int ks0 = C::kSplitK ? issuer * (C::kKSteps / 2) : 0;
      const int ks1 = C::kSplitK ? ks0 + C::kKSteps / 2 : C::kKSteps;
      const int at0 = ks0 >> 1, at1 = (ks1 + 1) >> 1;  // K groups (scale atoms) of those steps
      const uint32_t acc_slice = C::kSplitK ? issuer * C::kAccN : 0u;
      const uint32_t sf_col0 = C::kNumAcc * C::kAccCols;
      // shared-memory addresses of stage 0's parts; stage s adds s * kStageBytes
      const uint32_t a_addr0 = smem_u32(a_tile(0, 0));
      const uint32_t b_addr0 = smem_u32(b_tile(0));
      const uint32_t sfa_addr0 = smem_u32(sf_a(0, 0));
      const uint32_t sfb_addr0 = smem_u32(sf_b(0));
      // operand rows are kKBytes long (64-byte swizzle for 64, 128-byte for 128)
      auto kdesc = [](uint32_t saddr) {
        return C::kKBytes == 128 ? smem_desc_kmajor_sw128(saddr) : smem_desc_kmajor_sw64(saddr);
      };
      // a bounded wait whose outcome the whole warp shares
      auto wait_warp = [](uint64_t* bar, uint32_t parity, uint64_t limit) {
        return __shfl_sync(0xffffffffu, mbar_wait_bounded(bar, parity, limit) ? 1 : 0, 0) != 0;
      };
      int g = 0;
      bool err = false;
      for (int si = 0; si < sch.nseg && !err; ++si) {
        int u, kk0, kk1;
        bool whole;
        sch.seg(si, u, kk0, kk1, whole);
        const int b = si % C::kNumAcc;
        if (!wait_warp(&acce_bar[b], ((si / C::kNumAcc) & 1) ^ 1, p.wait_ns)) {
          if (leader) report_status(p.status, kStatusTimeoutMain);
          s_flags[0] = 1;
          break;
        }
        tc_fence_after();
        const uint32_t acc_base = tmem + b * C::kAccCols + acc_slice;
        bool seg_first = true;
        for (int kk = kk0; kk < kk1; ++kk, ++g) {
          const int s = g % C::kStages;
          const uint32_t ph = (g / C::kStages) & 1;
          if (!wait_warp(&full_bar[s], ph, p.wait_ns)) {
            if (leader) report_status(p.status, kStatusTimeoutMain);
            s_flags[0] = 1;
            err = true;
            break;
          }
          tc_fence_after();
          const uint32_t so = (uint32_t)s * C::kStageBytes;
          if constexpr (W16) {
            // bf16 x bf16: four K = 16 steps per 128-byte stage row, no scales; the
            // descriptors advance by adds (2 units of 16 bytes per 32-byte step)
            constexpr uint32_t idesc16 = idesc_bf16(kMTile, C::kN);
            const uint64_t bd0 = smem_desc_kmajor_sw128(b_addr0 + so);
            for (int j = j0; j < j1; ++j) {
              const uint64_t ad0 = smem_desc_kmajor_sw128(a_addr0 + so + j * C::kATileBytes);
#pragma unroll
              for (int ks = 0; ks < C::kKSteps; ++ks)
                mma_bf16_if(leader, acc_base + j * C::kAccN, ad0 + (uint64_t)(2 * ks), bd0 + (uint64_t)(2 * ks), idesc16,
                            (seg_first && ks == 0) ? 0u : 1u);
            }
            seg_first = false;
            mma_commit_if(leader, &empty_bar[s]);
            continue;
          }
          const uint32_t sfc = tmem + sf_col0 + s * C::kSfColsPerStage;
          // this issuer's copy of the B scale atoms (one shared copy with split K groups)
          const uint32_t sfb0 = sfc + 4 * C::kA * C::kAtoms + (C::kSplitK ? 0 : issuer * 4 * C::kNbAtoms * C::kAtoms);
          // scale atoms -> tensor memory (32 rows x 16 bytes, replicated to 4 lane quarters):
          // A tile j, K group a at columns 4 (j kAtoms + a); B atom (a, q) at 4 (a kNbAtoms + q)
          for (int j = j0; j < j1; ++j)
            for (int a = at0; a < at1; ++a) {
              const int i = j * C::kAtoms + a;
              tmem_cp_32x128b_warpx4_if(leader, sfc + 4 * i, smem_desc(sfa_addr0 + so + i * kSfAtomBytes, 0, 128, 0));
            }
          for (int i = at0 * C::kNbAtoms; i < at1 * C::kNbAtoms; ++i)
            tmem_cp_32x128b_warpx4_if(leader, sfb0 + 4 * i, smem_desc(sfb_addr0 + so + i * kSfAtomBytes, 0, 128, 0));
          if constexpr (C::kConcat) {
            for (int ks = ks0; ks < ks1; ++ks) {  // K = 64 steps: 32 bytes of every operand row
              if (kk * (C::kKStage / kMxBlock) + 2 * ks >= kblocks) break;  // both MX blocks are padding
              const int a = ks >> 1;                    // K group (scale atom) of this step
              const uint32_t idesc = idesc_mxf4(kMTile, C::kN, 2 * (ks & 1), 2 * (ks & 1));
              const uint64_t bdesc = kdesc(b_addr0 + so + 32 * ks);
              const uint32_t acc = seg_first ? 0u : 1u;
              for (int j = j0; j < j1; ++j) {
                const uint64_t adesc = kdesc(a_addr0 + so + j * C::kATileBytes + 32 * ks);
                mma_mxf4_if(leader, acc_base + j * C::kAccN, adesc, bdesc, idesc, sfc + 4 * (j * C::kAtoms + a),
                            sfb0 + 4 * a * C::kNbAtoms, acc);
              }
              seg_first = false;
            }
          } else {
            // One weight tile per issuer (j0) and one MMA per term.  At N = BM <= 128 an
            // MMA holds little tensor work, so the issuing thread's instructions set
            // the rate: the stage's descriptors are built once and advanced by adds
            // (the address field counts 16 bytes: 2 per 32-byte K step, BM * kKBytes / 16
            // per term), and the K steps and terms are unrolled with constant
            // instruction descriptors.
            static_assert(C::kA == 1 || C::kIssuers == 2, "one weight tile per issuer");
            const uint64_t ad0 = kdesc(a_addr0 + so + j0 * C::kATileBytes);
            const uint64_t bd0 = kdesc(b_addr0 + so);
            const uint32_t acc_j = acc_base + j0 * C::kAccN;
            const uint32_t sfa_j = sfc + 4 * (j0 * C::kAtoms);
            // K steps holding data: both MX blocks of a step past K are padding
            const int nsteps = min(C::kKSteps, (kblocks - kk * (C::kKStage / kMxBlock) + 1) >> 1);
#pragma unroll
            for (int ks = 0; ks < C::kKSteps; ++ks) {
              if (ks >= nsteps) break;
              const uint32_t idesc = idesc_mxf4(kMTile, C::kN, 2 * (ks & 1), 2 * (ks & 1));
#pragma unroll
              for (int t = 0; t < kTerms; ++t)
                mma_mxf4_if(leader, acc_j, ad0 + (uint64_t)(2 * ks),
                            bd0 + (uint64_t)((t * BM * C::kKBytes) / 16 + 2 * ks), idesc,
                            sfa_j + 4 * (ks >> 1), sfb0 + 4 * (ks >> 1) * C::kNbAtoms + (t * BM) / 32,
                            (seg_first && ks == 0 && t == 0) ? 0u : 1u);
            }
            seg_first = false;
          }
          mma_commit_if(leader, &empty_bar[s]);  // frees the stage once both issuers' MMAs have read it
        }
        if (!err) mma_commit_if(leader, &accf_bar[b]);
      }
      // every tensor-core operation this warp issued (MMAs, scale copies) completes
      // before the CTA frees its tensor memory and exits (long limit, as above)
      mma_commit_if(leader, drain_bar);
      wait_warp(drain_bar, 0, kWaitLimit);
    }
  } else if ((warp >= 2 && warp < 6) || (C::kEpiGroups == 2 && warp >= 7 && warp < 11)) {
    // ------------------------------------------------------------ epilogue
    pdl_wait();  // h (down) comes from the immediately preceding kernel
    const int eg = warp < 6 ? 0 : 1;       // epilogue group: warps 2-5, or 7-10
    const int q = warp & 3;                // tensor-memory lane quarter of this warp
    const int m = q * 32 + lane;           // row of the 128-row tile
    const int et = threadIdx.x - (eg == 0 ? 64 : 224);  // 0..127 within the group
    float* s_xpose = reinterpret_cast<float*>(epi_smem + eg * C::kEpiGroupBytes);
    int* s_rowa = reinterpret_cast<int*>(s_xpose + 16 * kMTile);
    float* s_roww = reinterpret_cast<float*>(s_rowa + C::kMetaRows);
    auto epi_bar = [eg]() { asm volatile("bar.sync %0, 128;" ::"r"(1 + eg) : "memory"); };
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    const int i_pad = (p.I + 63) / 64 * 64;  // h features written (zeros past I)
    const bool split_live = p.K > 2 * 2 * kMxBlock;  // the second issuer's K group holds data
    for (int si = 0; si < sch.nseg; ++si) {
      int u, kk0, kk1, tile, mt;
      bool whole;
      sch.seg(si, u, kk0, kk1, whole);
      const int b = si % C::kNumAcc;
      map_unit(u, num_tiles, p.mt, p.group_tiles, tile, mt);
      const TileEntry te = load_tile(p.tiles + tile);
      const int nrows = te.n_rows;
      const int feat = mt * kMTile + m;
      if constexpr (!GATEUP) {
        // row metadata of the tile, staged before the accumulator is ready
        for (int r = et; r < nrows; r += 128) {
          const int a = __ldcg(p.perm + te.row_begin + r);
          s_rowa[r] = a;
          s_roww[r] = __ldcg(p.topk_w + a);
        }
      }
      const bool ok = mbar_wait_bounded(&accf_bar[b], (si / C::kNumAcc) & 1, p.wait_ns);
      if (!ok) {
        report_status(p.status, kStatusTimeoutEpi);
        s_flags[0] = 1;
        break;
      }
      tc_fence_after();
      epi_bar();  // row metadata visible
      const uint32_t acc_addr = tmem + lane_off + b * C::kAccCols;

      // h = silu(g) * u of the 16 token columns from c0 (this thread's feature row m),
      // computed for the tile's real tokens only (zero past them or past I)
      auto silu_mul = [&](int c0, const float* va, const float* vb, float* h) {
        const bool fvalid = feat < p.I;
#pragma unroll
        for (int j = 0; j < 16; ++j) h[j] = (fvalid && c0 + j < nrows) ? silu_f(va[j]) * vb[j] : 0.f;
      };
      // h of 16 token columns -> shared memory, transposed so that threads hold runs of
      // features of one token column, then encoded as kTerms E2M1 terms into the down
      // GEMM's B layout
      auto encode_h = [&](int c0, const float* h) {
#pragma unroll
        for (int j = 0; j < 16; ++j)
          if (c0 + j < nrows) s_xpose[j * kMTile + m] = h[j];
        epi_bar();
        // Each column's 4 MX blocks of 32 features are encoded by 128 / V threads, V
        // values each (32 / V threads per block), with V the smallest of 4, 8 and 16
        // whose 128-thread cover reaches the chunk's real columns: a tile with few
        // tokens gives each thread a shorter dependent chain of terms.
        const int live = min(16, nrows - c0);
        uint8_t* sf = p.h_sf + ((size_t)tile * p.kg_out + mt) * (kSfAtomBytes * act_sf_atoms(BM));
        auto encode = [&](auto v_tag) {
          constexpr int V = decltype(v_tag)::value;
          constexpr int kTpb = 32 / V;    // threads per MX block
          constexpr int kTpc = 4 * kTpb;  // threads per column
          const int j = et / kTpc, qb = (et % kTpc) / kTpb, sub = et % kTpb;
          const int r = c0 + j;
          float vv[V];
          const float4* src = reinterpret_cast<const float4*>(s_xpose + j * kMTile + qb * 32 + sub * V);
#pragma unroll
          for (int i = 0; i < V / 4; ++i) {
            const float4 f4 = src[i];
            vv[4 * i] = f4.x;
            vv[4 * i + 1] = f4.y;
            vv[4 * i + 2] = f4.z;
            vv[4 * i + 3] = f4.w;
          }
          const int feat0 = mt * kMTile + qb * 32 + sub * V;
#pragma unroll
          for (int t = 0; t < kTerms; ++t) {
            float amax = 0.f;
#pragma unroll
            for (int i = 0; i < V; ++i) amax = fmaxf(amax, fabsf(vv[i]));
#pragma unroll
            for (int d = 1; d < kTpb; d <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, d));
            const int pe = mx_e2m1_exponent(amax);
            const float inv = pow2_int(-pe), sc = pow2_int(pe);
            uint32_t w[(V + 7) / 8] = {};
#pragma unroll
            for (int i = 0; i < V / 2; ++i) {
              const uint32_t pair = f32x2_to_e2m1x2(vv[2 * i] * inv, vv[2 * i + 1] * inv);
              const float2 q = e2m1x2_to_f32x2(pair);
              vv[2 * i] -= q.x * sc;
              vv[2 * i + 1] -= q.y * sc;
              w[i >> 2] |= pair << (8 * (i & 3));
            }
            // the column's 4 blocks start at lanes base, base + kTpb, ...: pack the exponents
            const uint32_t e8 = static_cast<uint32_t>(pe + 127);
            const int base = lane & ~(kTpc - 1);
            const uint32_t word = __shfl_sync(0xffffffffu, e8, base) |
                                  (__shfl_sync(0xffffffffu, e8, base + kTpb) << 8) |
                                  (__shfl_sync(0xffffffffu, e8, base + 2 * kTpb) << 16) |
                                  (__shfl_sync(0xffffffffu, e8, base + 3 * kTpb) << 24);
            if (r < nrows) {
              if (feat0 < i_pad) {
                uint8_t* dst = p.h_q + act_offset(tile, t, r, feat0, p.max_tiles, BM);
                if constexpr (V == 16) *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[1]);
                else if constexpr (V == 8) *reinterpret_cast<uint32_t*>(dst) = w[0];
                else *reinterpret_cast<uint16_t*>(dst) = static_cast<uint16_t>(w[0]);
              }
              if (et % kTpc == 0) *reinterpret_cast<uint32_t*>(sf + sf_atom_offset(act_row(t, r, BM), 0)) = word;
            }
          }
        };
        if constexpr (BM == 16) {
          if (live <= 4)
            encode(std::integral_constant<int, 4>{});
          else if (live <= 8)
            encode(std::integral_constant<int, 8>{});
          else
            encode(std::integral_constant<int, 16>{});
        } else {
          encode(std::integral_constant<int, 16>{});  // larger tiles: full chunks but the last
        }
        epi_bar();  // s_xpose reused by the next chunk
      };

      // the math of 16 token columns starting at c0, given g/u (gate/up) or y (down)
      auto consume = [&](int c0, const float* va, const float* vb) {
        if constexpr (GATEUP && W16) {
          // h = silu(g) * u -> shared memory (transposed), then bf16 rows of h in the
          // down GEMM's B layout: thread (column j, 16 features qb) stores two 16-byte chunks
          const bool fvalid = feat < p.I;
#pragma unroll
          for (int j = 0; j < 16; ++j) s_xpose[j * kMTile + m] = fvalid ? silu_f(va[j]) * vb[j] : 0.f;
          epi_bar();
          const int j = et >> 3, qb = et & 7;
          const int r = c0 + j, f0 = mt * kMTile + qb * 16;
          if (r < nrows && f0 < p.I) {
            const float4* src = reinterpret_cast<const float4*>(s_xpose + j * kMTile + qb * 16);
            uint32_t w[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float4 f4 = src[i];
              w[2 * i] = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(f4.x)) |
                         ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(f4.y)) << 16);
              w[2 * i + 1] = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(f4.z)) |
                             ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(f4.w)) << 16);
            }
            *reinterpret_cast<uint4*>(p.h_q + act16_offset(tile, r, f0, p.max_tiles, BM)) =
                make_uint4(w[0], w[1], w[2], w[3]);
            *reinterpret_cast<uint4*>(p.h_q + act16_offset(tile, r, f0 + 8, p.max_tiles, BM)) =
                make_uint4(w[4], w[5], w[6], w[7]);
          }
          epi_bar();  // s_xpose reused by the next chunk
        } else if constexpr (GATEUP) {
          float h[16];
          silu_mul(c0, va, vb, h);
          encode_h(c0, h);
        } else {
          // output features: M tile mt, or the pair 2 mt, 2 mt + 1 (va, vb)
          const int fa = (MPAIR ? 2 * mt : mt) * kMTile + m;
          const int fb = fa + kMTile;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int r = c0 + j;
            if (r < nrows) {
              float* slot = p.slots + (size_t)s_rowa[r] * p.H;
              if (fa < p.H) slot[fa] = s_roww[r] * va[j];
              if (MPAIR && fb < p.H) slot[fb] = s_roww[r] * vb[j];
            }
          }
        }
      };

      if constexpr (C::kLoadAll) {
        // whole accumulator -> registers, release it to the MMA warp, then compute
        float acc[C::kAccCols];
#pragma unroll
        for (int c0 = 0; c0 < C::kAccCols; c0 += 16) {
          uint32_t r[16];
          tmem_ld_32x32b_x16(acc_addr + c0, r);
#pragma unroll
          for (int j = 0; j < 16; ++j) acc[c0 + j] = __uint_as_float(r[j]);
        }
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(&acce_bar[b]);
        // values: add the term columns when the terms share one MMA (token-major
        // columns: token c's terms are columns 4c .. 4c + 3)
        float vals[C::kVals];
#pragma unroll
        for (int j = 0; j < C::kA; ++j)
#pragma unroll
          for (int c = 0; c < BM; ++c) {
            // split K groups: the two slices hold partial sums of the same products (the
            // second one only when K reaches past the first K group of 128)
            auto col = [&](int i) {
              return C::kSplitK ? acc[j * C::kAccN + i] + (split_live ? acc[C::kAccN + i] : 0.f)
                                : acc[j * C::kAccN + i];
            };
            float v;
            if constexpr (C::kConcat) {
              v = col(kTerms * c);
#pragma unroll
              for (int t = 1; t < kTerms; ++t) v += col(kTerms * c + t);
            } else {
              v = col(c);
            }
            vals[j * BM + c] = v;
          }
#pragma unroll
        for (int c0 = 0; c0 < BM; c0 += 16)
          if (c0 < nrows) consume(c0, vals + c0, C::kA > 1 ? vals + BM + c0 : nullptr);
      } else {
        // accumulator too large for registers (per-term MMAs): 16 columns at a time,
        // the groups taking alternate chunks
        if constexpr (GATEUP && !W16) {
          // h of all this thread's chunks first (BM / 16 / groups chunks of 16 values),
          // then the accumulator goes back to the MMA warps, and the transposes and the
          // long four-term encode run while the next unit's MMAs do
          constexpr int kChunks = BM / 16 / C::kEpiGroups;
          float hreg[kChunks][16];
#pragma unroll
          for (int i = 0; i < kChunks; ++i) {
            const int c0 = 16 * (eg + C::kEpiGroups * i);
            if (c0 < nrows) {
              uint32_t rg[16], ru[16];
              float va[16], vb[16];
              tmem_ld_32x32b_x16(acc_addr + c0, rg);
              tmem_ld_32x32b_x16(acc_addr + C::kAccN + c0, ru);
              tmem_wait_ld();
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                va[j] = __uint_as_float(rg[j]);
                vb[j] = __uint_as_float(ru[j]);
              }
              silu_mul(c0, va, vb, hreg[i]);
            }
          }
          tc_fence_before();
          mbar_arrive(&acce_bar[b]);
#pragma unroll
          for (int i = 0; i < kChunks; ++i) {
            const int c0 = 16 * (eg + C::kEpiGroups * i);
            if (c0 < nrows) encode_h(c0, hreg[i]);
          }
        } else if constexpr (!GATEUP && !W16) {
          // down: all this thread's chunks into registers, the accumulator back to the
          // MMA warps, then the weighted slot stores
          constexpr int kChunks = BM / 16 / C::kEpiGroups;
          float ya[kChunks][16], yb[kChunks][16];
#pragma unroll
          for (int i = 0; i < kChunks; ++i) {
            const int c0 = 16 * (eg + C::kEpiGroups * i);
            if (c0 < nrows) {
              uint32_t rg[16], ru[16];
              tmem_ld_32x32b_x16(acc_addr + c0, rg);
              if (C::kA > 1) tmem_ld_32x32b_x16(acc_addr + C::kAccN + c0, ru);
              tmem_wait_ld();
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                ya[i][j] = __uint_as_float(rg[j]);
                yb[i][j] = C::kA > 1 ? __uint_as_float(ru[j]) : 0.f;
              }
            }
          }
          tc_fence_before();
          mbar_arrive(&acce_bar[b]);
#pragma unroll
          for (int i = 0; i < kChunks; ++i) {
            const int c0 = 16 * (eg + C::kEpiGroups * i);
            if (c0 < nrows) consume(c0, ya[i], yb[i]);
          }
        } else {
          for (int c0 = 16 * eg; c0 < BM; c0 += 16 * C::kEpiGroups) {
            if (c0 >= nrows) break;
            uint32_t rg[16], ru[16];
            float va[16], vb[16];
            tmem_ld_32x32b_x16(acc_addr + c0, rg);
            if (C::kA > 1) tmem_ld_32x32b_x16(acc_addr + C::kAccN + c0, ru);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              va[j] = __uint_as_float(rg[j]);
              vb[j] = C::kA > 1 ? __uint_as_float(ru[j]) : 0.f;
            }
            consume(c0, va, vb);
          }
          tc_fence_before();
          mbar_arrive(&acce_bar[b]);
        }
      }

      epi_bar();  // row metadata is reused by the next segment
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, C::kTmemCols);
}

// ------------------------------------------------------------------ host launchers
template <int BM, bool GATEUP, bool MPAIR, bool W16>
static cudaError_t launch_gemm_t(const GemmParams& p, cudaStream_t stream) {
  using C = GemmCfg<BM, GATEUP, MPAIR, W16>;
  auto kern = moe_gemm_kernel<BM, GATEUP, MPAIR, W16>;
  static SmemOptIn opt_in;
  const cudaError_t e = opt_in.ensure(kern, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(p.grid), dim3(C::kThreads), C::kSmemBytes, stream, p);
}

template <bool GATEUP, bool MPAIR, bool W16>
static cudaError_t launch_gemm(const GemmParams& p, cudaStream_t stream) {
  switch (p.bm) {
    case 16: return launch_gemm_t<16, GATEUP, MPAIR, W16>(p, stream);
    case 64: return launch_gemm_t<64, GATEUP, MPAIR, W16>(p, stream);
    case 128: return launch_gemm_t<128, GATEUP, MPAIR, W16>(p, stream);
    case 256:  // bf16 only (no scale columns), unpaired down: the accumulators fit tensor memory
      if constexpr (W16 && !MPAIR) return launch_gemm_t<256, GATEUP, MPAIR, W16>(p, stream);
      return cudaErrorInvalidValue;
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_gateup(const GemmParams& p, cudaStream_t stream) {
  return p.w16 ? launch_gemm<true, false, true>(p, stream) : launch_gemm<true, false, false>(p, stream);
}
cudaError_t launch_down(const GemmParams& p, cudaStream_t stream) {
  if (p.w16) return p.m_pair ? launch_gemm<false, true, true>(p, stream) : launch_gemm<false, false, true>(p, stream);
  return p.m_pair ? launch_gemm<false, true, false>(p, stream) : launch_gemm<false, false, false>(p, stream);
}

}  // namespace moe
