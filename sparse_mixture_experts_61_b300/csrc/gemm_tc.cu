// GEMMs on the 5th-generation tensor cores (tcgen05, sm_103a): the two expert GEMMs
// of the expert FFN and the router contraction.
//
//   expert FFN ("MoE mixture-of-experts routing mechanism: principles and sparse
//   activation", Expert.forward = w2(silu(w1(x))) with nn.Linear biases), run as one
//   ragged grouped GEMM per layer -- the job "Breaking the MoE trilemma" 3.3 gives
//   _grouped_ffn, with every expert's token group handled by one kernel launch:
//       out[r, n] = act( sum_c X[r, c] * W[g][n][c] + bias[g][n] ),  r in group g's rows
//   router (gating formula, x . W_g):  logits[t, e] = sum_c x[t, c] * W_g[e, c] + b[e].
//
// Both kernels share one warp-specialised pipeline (one persistent CTA per SM):
//  * warp 0: TMA producer.  128-byte-swizzled K-major tiles, 64 bf16 deep.
//  * warp 1: allocates TMEM (two fp32 accumulators) and issues tcgen05.mma from one
//    thread, committing each shared-memory stage back to the producer and each
//    finished accumulator to the epilogue.
//  * warps 2-5: epilogue, draining TMEM with tcgen05.ld while the next tile's main
//    loop runs in the other accumulator (warps 2-9 in the row-tile expert GEMM, two
//    per TMEM lane quadrant, each taking half of the tile's columns).
//  * Every wait is bounded (common.cuh); on a timeout the CTA records
//    MOE_DEVERR_TIMEOUT, lets its own TMA copies and MMAs land, frees TMEM, returns.
//
// Small expert groups use the "weights as M" orientation: the MMA's M = 128 side is a
// block of 128 weight rows (output features), which always fills the tile, and its N
// side is a block of one expert's token rows, set per tile in the instruction
// descriptor.  An expert's n rows are cut into nt = ceil(n / TB) equal blocks of
// ceil(n / nt) rows rounded up to 16, so a ragged group costs at most 15 padded token
// columns per block.  Every CTA loads its own weight rows and token rows with plain
// TMA tile loads.  The (tile, k-block) iterations of the whole layer are divided evenly
// over the CTAs (a stream-K split): a CTA's share may start or end inside a tile, so a
// few tiles are computed in pieces by consecutive CTAs.  Each piece parks its fp32 sums
// in the workspace; the CTA whose piece lands last adds the pieces in k order (a fixed
// order, so results do not depend on timing) and runs the epilogue.  This keeps every
// SM busy to the end whether the layer has fewer tiles than SMs (a Switch layer's
// second GEMM: 72 tiles of 64 k-blocks) or a few more than a multiple of them.  The
// tile list is derived on the device from the group offsets: the kept-row count never
// goes to the host.
//
// Large groups use row tiles: 128 token rows x 256 weight rows, tokens as M.
// The router keeps tokens as M (128 rows per tile) and the E experts as N.

#include "tc_pipe.cuh"

namespace moe {
namespace {

// ------------------------------------------------------------- expert FFN GEMM
// A = weight block [128 x 64] of W[g] (3-D map over [G, N, K]); B = token block of
// up to TB rows, loaded as boxes of tok_box(TB) rows (2-D map over [rows_alloc, K]);
// D[128 x ntok] in TMEM, lane = output feature, column = token.
// Token box height: the whole token tile up to 64 rows.  Fewer, larger copies per
// k-block measured faster than exact-fit ones: 64-row boxes took the 64-token decode
// layer's expert GEMMs from 711 to 706 us (bitwise the same), and 16-row boxes made the
// Switch layer's 4% slower than 32-row ones despite loading fewer padding rows.
constexpr int tok_box(int tb) { return tb < 64 ? tb : 64; }
// Fewest iterations (k-blocks) in a CTA's share of the split; a layer with fewer than
// this many per CTA runs on fewer CTAs.
constexpr int kMinSplitKb = 8;
// What parking and adding up a split tile's pieces costs, in k-block iterations: the
// split is taken only when it shortens the longest CTA's share by more than this and
// by at least an eighth.  Measured on the Switch layer: parking a piece and counting it
// in takes ~1 us, and the CTA that finishes a tile spends 2-4 us per 32 token columns
// on L2 round trips, ~9 us in all, about 24-32 k-blocks of a saturated main loop (a
// split of its 72-tile second GEMM ran 12 us slower than whole tiles on 72 SMs; on the
// 64-token decode layer, whose second GEMM has 4.1 waves of whole tiles, it is 4.5%
// faster).
constexpr int kSplitCostKb = 32;
// Pieces whose parked sums the finishing CTA loads at once.
constexpr int kReduceBatch = 2;

// The even division of `total` (tile, k-block) iterations over `parts` CTAs: CTA c
// runs iterations [begin(c), begin(c + 1)).
struct SplitK {
  int64_t total;
  int parts;
  __device__ __forceinline__ int64_t begin(int c) const { return total * c / parts; }
  // The CTA whose share holds iteration `it`: the largest c with begin(c) <= it, which
  // never has an empty share.
  __device__ __forceinline__ int owner(int64_t it) const {
    return static_cast<int>(((it + 1) * parts + total - 1) / total - 1);
  }
  __device__ __forceinline__ bool busy(int c) const { return begin(c) < begin(c + 1); }
};

template <int TB, int STAGES, int EPI, bool GATHER, bool TOP1>
__global__ void __launch_bounds__(TC_THREADS, 1)
    tc_ffn_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                  const GemmArgs p) {
  constexpr int TOK_BOX = tok_box(TB);
  static_assert(TB >= TOK_BOX && TB <= 128 && (TB & (TB - 1)) == 0,
                "TB: power of two in [32, 128]");
  static_assert(EPI == EPI_BIAS_SILU || EPI == EPI_BIAS, "expert epilogues only");
  constexpr uint32_t kTmemCols = 2 * TB;
  constexpr uint32_t kWeightBytes = TILE_M * TC_BK * 2;
  constexpr uint32_t kBoxBytes = TOK_BOX * TC_BK * 2;
  constexpr int64_t kPartFloats = int64_t{TILE_M} * TB;  // one parked piece
  constexpr uint32_t kRowBytes = TC_BK * 2;              // one token row of a k-block
  using Smem = PipeSmem<TILE_M * TC_BK * 2, TB * TC_BK * 2, STAGES>;
  Smem& S = smem_aligned<Smem>();
  // Gathered token rows: the current piece's token ids, after the pipeline state in the
  // dynamic shared memory (allocated only for a gathering launch, so that the default
  // launch's footprint is unchanged).
  int* s_tok = reinterpret_cast<int*>(
      (reinterpret_cast<uintptr_t>(&S) + sizeof(Smem) + 15) & ~static_cast<uintptr_t>(15));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.G;
  pipe_prologue<Smem, STAGES>(S, kTmemCols, p, G, TB, &tmW, &tmX);

  const int MB = (p.N + TILE_M - 1) / TILE_M;  // weight blocks per group
  const int KB = (p.K + TC_BK - 1) / TC_BK;
  const int64_t ntiles = static_cast<int64_t>(S.pref[G]) * MB;
  const int grid = static_cast<int>(gridDim.x), cta = static_cast<int>(blockIdx.x);
  SplitK sk;
  sk.total = ntiles * KB;
  {
    const int64_t by_size = sk.total / kMinSplitKb;
    sk.parts = static_cast<int>(by_size < 1 ? 1 : by_size < grid ? by_size : grid);
  }
  // Whole tiles round-robin (the longest share is ceil(tiles / grid) tiles), or the
  // even split of the iterations; every CTA takes the same decision.
  const int64_t longest_whole = (ntiles + grid - 1) / grid * KB;
  const int64_t longest_split = (sk.total + sk.parts - 1) / sk.parts;
  const bool split = sk.parts > 1 && longest_split + kSplitCostKb < longest_whole &&
                     (longest_whole - longest_split) * 8 >= longest_whole;
  int64_t it0 = 0, it1 = 0;
  int npieces = 0;
  if (split) {
    it0 = cta < sk.parts ? sk.begin(cta) : 0;
    it1 = cta < sk.parts ? sk.begin(cta + 1) : 0;
    npieces = it1 > it0 ? static_cast<int>((it1 - 1) / KB - it0 / KB + 1) : 0;
  } else {
    npieces = ntiles > cta ? static_cast<int>((ntiles - cta + grid - 1) / grid) : 0;
  }
  volatile int* abort = &S.abort;

  struct Coord {
    int g, n0, ntok, nbox, kb0, kb1;
    uint32_t bytes;
    int64_t row0, row_end, tile;
  };
  // Piece q of this CTA: the tile it belongs to and its k-blocks [kb0, kb1).
  auto decode = [&](int q) {
    Coord c;
    if (split) {
      c.tile = it0 / KB + q;
      const int64_t t0 = c.tile * KB;
      c.kb0 = static_cast<int>((t0 > it0 ? t0 : it0) - t0);
      c.kb1 = static_cast<int>((t0 + KB < it1 ? t0 + KB : it1) - t0);
    } else {
      c.tile = cta + static_cast<int64_t>(q) * grid;
      c.kb0 = 0;
      c.kb1 = KB;
    }
    const int tile = static_cast<int>(c.tile);
    c.g = find_group(S.pref, G, MB, tile);
    const int nt = S.pref[c.g + 1] - S.pref[c.g];
    const int local = tile - S.pref[c.g] * MB;
    c.n0 = (local / nt) * TILE_M;
    const int64_t base = p.offsets[c.g], end = p.offsets[c.g + 1];
    const int64_t bsz = (((end - base) + nt - 1) / nt + 15) & ~int64_t{15};
    c.row0 = base + (local % nt) * bsz;
    c.row_end = c.row0 + bsz < end ? c.row0 + bsz : end;
    c.ntok = static_cast<int>((c.row_end - c.row0 + 15) & ~int64_t{15});
    c.nbox = (c.ntok + TOK_BOX - 1) / TOK_BOX;
    c.bytes = kWeightBytes + (GATHER ? static_cast<uint32_t>(c.ntok) * kRowBytes
                                     : static_cast<uint32_t>(c.nbox) * kBoxBytes);
    return c;
  };

  if (warp == 0) {
    if constexpr (GATHER) {
      // Token rows straight from x: the piece's token ids are fetched by the whole warp
      // (the block's padding rows repeat its last token; an id outside [0, rows) is
      // flagged and read as token 0), then four rows of x per gather.
      run_producer_warp<STAGES>(
          S, 0, 1, npieces, decode,
          [&](const Coord& c, int ln) {
            for (int i = ln; i < c.ntok; i += 32) {
              const int64_t r = c.row0 + i < c.row_end ? c.row0 + i : c.row_end - 1;
              int t = p.gather_rows[r];
              if (t < 0 || t >= p.gather_src_rows) {
                raise_flag(p.flags, MOE_DEVERR_BAD_ROW);
                t = 0;
              }
              s_tok[i] = t;
            }
          },
          [&](const Coord& c, int kb, uint32_t sa, uint32_t sb, uint32_t bar) {
            tma_load_3d(sa, &tmW, bar, kb * TC_BK, c.n0, c.g);
            for (int j = 0; j < c.ntok; j += 4)
              tma_gather4(sb + j * kRowBytes, &tmX, bar, kb * TC_BK, s_tok[j], s_tok[j + 1],
                          s_tok[j + 2], s_tok[j + 3]);
          },
          abort, p.flags);
    } else if (lane == 0) {
      run_producer<STAGES>(
          S, 0, 1, npieces, decode,
          [&](const Coord& c, int kb, uint32_t sa, uint32_t sb, uint32_t bar) {
            tma_load_3d(sa, &tmW, bar, kb * TC_BK, c.n0, c.g);
            for (int j = 0; j < c.nbox; ++j)
              tma_load_2d(sb + j * kBoxBytes, &tmX, bar, kb * TC_BK,
                          static_cast<int>(c.row0) + j * TOK_BOX);
          },
          abort, p.flags);
    }
  } else if (warp == 1) {
    if (lane == 0)
      run_mma<STAGES, TB>(S, 0, 1, npieces, S.tmem_base, decode,
                          [](const Coord& c) { return bf16_idesc(TILE_M, c.ntok); }, abort,
                          p.flags);
  } else {
    const int quad = warp & 3;  // TMEM lanes this warp may read: 32*quad .. 32*quad+31
    if constexpr (TOP1 && EPI == EPI_BIAS_SILU) {
      // Top-1 combine, first part: zero the layer-output rows of the tokens whose slot was
      // dropped (GEMM 2 writes every other token's row), one warp per token, while the
      // first tiles' operands stream in.
      // A warp takes 32 consecutive tokens at a time: their slots are read one per lane in
      // a single round trip, then the dropped tokens' rows are written.
      const int nvec = p.comb_cols / 8;
      uint4* y = static_cast<uint4*>(p.comb_out);
      const int64_t nw = static_cast<int64_t>(grid) * (TC_THREADS / 32 - 2) * 32;
      for (int64_t t0 = (static_cast<int64_t>(cta) * (TC_THREADS / 32 - 2) + (warp - 2)) * 32;
           t0 < p.comb_rows; t0 += nw) {
        const int64_t t = t0 + lane;
        unsigned drop = __ballot_sync(0xffffffffu, t < p.comb_rows && p.comb_slot[t] < 0);
        while (drop) {
          const int i = __ffs(drop) - 1;
          drop &= drop - 1;
          uint4* row = y + (t0 + i) * nvec;
          for (int v = lane; v < nvec; v += 32) row[v] = make_uint4(0u, 0u, 0u, 0u);
        }
      }
    }
    int acc = 0;
    uint32_t aph = 0;
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out);
    const __nv_bfloat16* bias = static_cast<const __nv_bfloat16*>(p.bias);
    for (int q = 0; q < npieces; ++q) {
      const Coord c = decode(q);
      const int n = c.n0 + quad * 32 + lane;
      const bool n_ok = n < p.N;
      const float b = (bias && n_ok) ? __bfloat162float(bias[static_cast<int64_t>(c.g) * p.N + n])
                                     : 0.f;
      // Top-1 combine: the tokens and gate weights of the tile's rows, one per lane for each
      // 32-row chunk, read before the accumulator is ready.
      int tok[TB / 32];
      float gate[TB / 32];
      if constexpr (TOP1 && EPI == EPI_BIAS) {
#pragma unroll
        for (int j = 0; j < TB / 32; ++j) {
          const int64_t r = c.row0 + 32 * j + lane;
          tok[j] = r < c.row_end ? p.comb_token[r] : -1;
        }
#pragma unroll
        for (int j = 0; j < TB / 32; ++j) {
          if (tok[j] >= p.comb_rows || (tok[j] < 0 && c.row0 + 32 * j + lane < c.row_end)) {
            raise_flag(p.flags, MOE_DEVERR_BAD_ROW);
            tok[j] = -1;
          }
          gate[j] = tok[j] >= 0 ? p.comb_w[tok[j]] : 0.f;
        }
      }
      const bool got = mbar_wait_bounded(smem_u32(&S.tfull[acc]), aph, abort, p.flags);
      if (!__all_sync(0xffffffffu, got)) break;  // the warp-collective loads need every lane
      tc_fence_after();
      const uint32_t t_row = S.tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                             static_cast<uint32_t>(acc * TB);
      const int nrows = static_cast<int>(c.row_end - c.row0);
      // Bias, activation and bf16 store of feature n for token columns [col, col + 32).
      auto store = [&](int col, const float(&v)[32]) {
        if constexpr (TOP1 && EPI == EPI_BIAS) {
          // Top-1 combine: row i's output goes to its token's row of the layer output,
          // scaled by the token's gate weight the way the combine scales one slot.  The
          // 32 rows' tokens and weights (read ahead, one per lane) are shared by shuffles.
          int tk = -1;
          float gw = 0.f;
#pragma unroll
          for (int j = 0; j < TB / 32; ++j)
            if (col == 32 * j) {
              tk = tok[j];
              gw = gate[j];
            }
          __nv_bfloat16* y = static_cast<__nv_bfloat16*>(p.comb_out);
          // Eight rows' tokens and weights are shuffled out together, then stored, so the
          // shuffles' latency is not paid row by row.
#pragma unroll
          for (int i0 = 0; i0 < 32; i0 += 8) {
            int t8[8];
            float w8[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              t8[u] = __shfl_sync(0xffffffffu, tk, i0 + u);
              w8[u] = __shfl_sync(0xffffffffu, gw, i0 + u);
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              if (n_ok && t8[u] >= 0) {
                const float yp = __bfloat162float(__float2bfloat16_rn(v[i0 + u] + b));
                y[static_cast<int64_t>(t8[u]) * p.N + n] = __float2bfloat16_rn(fmaf(w8[u], yp, 0.f));
              }
            }
          }
          return;
        }
        if (!n_ok) return;
        __nv_bfloat16* o = out + (c.row0 + col) * p.N + n;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          if (col + i < nrows) {
            float x = v[i] + b;
            if (EPI == EPI_BIAS_SILU) {
              if (p.pre_out)
                static_cast<__nv_bfloat16*>(p.pre_out)[(o - out) + static_cast<int64_t>(i) * p.N] =
                    __float2bfloat16_rn(x);
              x = silu(x);
            }
            o[static_cast<int64_t>(i) * p.N] = __float2bfloat16_rn(x);
          }
        }
      };
      if (c.kb0 == 0 && c.kb1 == KB) {
#pragma unroll 1
        for (int col = 0; col < c.ntok; col += 32) {
          float v[32];
          tmem_ld_32cols(t_row + col, v);
          tc_wait_ld();
          store(col, v);
        }
        tc_fence_before();
        mbar_arrive(smem_u32(&S.tempty[acc]));
      } else {
        // A piece of a split tile.  Park its sums ([token][feature] within the piece's
        // slot: slot 1 for a tile's first piece, slot 0 for a later one; a CTA holds at
        // most one of each), then count the piece in on the tile's counter (one per
        // lane quadrant, indexed by the CTA holding the tile's first piece).
        const int64_t t0 = c.tile * KB;
        const int first = sk.owner(t0), last = sk.owner(t0 + KB - 1);
        float* mine = p.sk_part + (static_cast<int64_t>(cta) * 2 + (c.kb0 > 0 ? 0 : 1)) * kPartFloats +
                      quad * 32 + lane;
#pragma unroll 1
        for (int col = 0; col < c.ntok; col += 32) {
          float v[32];
          tmem_ld_32cols(t_row + col, v);
          tc_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (col + i < nrows) mine[static_cast<int64_t>(col + i) * TILE_M] = v[i];
        }
        tc_fence_before();
        mbar_arrive(smem_u32(&S.tempty[acc]));  // the accumulator is free again
        __threadfence();
        __syncwarp();
        int pieces = 0;
        for (int cc = first; cc <= last; ++cc) pieces += sk.busy(cc) ? 1 : 0;
        int* ctr = p.sk_ctr + first * 4 + quad;
        int arrived = 0;
        if (lane == 0) arrived = atomicAdd(ctr, 1);
        arrived = __shfl_sync(0xffffffffu, arrived, 0);
        if (arrived == pieces - 1) {
          // Every other piece has landed: add them in k order and finish the tile.
          // The loads of kReduceBatch pieces are issued together, then added in order.
          if (lane == 0) atomicExch(ctr, 0);  // ready for the next launch
          __threadfence();
#pragma unroll 1
          for (int col = 0; col < nrows; col += 32) {
            float v[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = 0.f;
            bool lead = true;
#pragma unroll 1
            for (int cc0 = first; cc0 <= last; cc0 += kReduceBatch) {
              float x[kReduceBatch][32];
              bool use[kReduceBatch];
#pragma unroll
              for (int u = 0; u < kReduceBatch; ++u) {
                const int cc = cc0 + u;
                use[u] = cc <= last && sk.busy(cc);
                const float* src =
                    p.sk_part + (static_cast<int64_t>(cc) * 2 + (cc == first ? 1 : 0)) * kPartFloats +
                    quad * 32 + lane;
#pragma unroll
                for (int i = 0; i < 32; ++i)
                  x[u][i] = (use[u] && col + i < nrows)
                                ? __ldcg(src + static_cast<int64_t>(col + i) * TILE_M)
                                : 0.f;
              }
#pragma unroll
              for (int u = 0; u < kReduceBatch; ++u) {
                if (!use[u]) continue;
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = lead ? x[u][i] : v[i] + x[u][i];
                lead = false;
              }
            }
            store(col, v);
          }
        }
      }
      acc ^= 1;
      if (acc == 0) aph ^= 1u;
    }
  }
  pipe_teardown(S, kTmemCols);
}

// Bias (and SiLU) of 32 accumulator columns of one row, packed to bf16: v holds the fp32
// accumulators, bias (or null) the 32 columns' biases; pre receives the packed
// pre-activation when the epilogue is SiLU.
template <int EPI>
__device__ __forceinline__ void bias_act_32(const float (&v)[32], const uint4 (&bias)[4],
                                           bool has_bias, uint4 (&packed)[4], uint4 (&pre)[4]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    float b[8];
    if (has_bias) {
      const __nv_bfloat162* bh = reinterpret_cast<const __nv_bfloat162*>(&bias[q]);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(bh[i]);
        b[2 * i] = f.x;
        b[2 * i + 1] = f.y;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) b[i] = 0.f;
    }
    __nv_bfloat162* ph = reinterpret_cast<__nv_bfloat162*>(&packed[q]);
    __nv_bfloat162* pp = reinterpret_cast<__nv_bfloat162*>(&pre[q]);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float x0 = v[8 * q + 2 * i] + b[2 * i];
      float x1 = v[8 * q + 2 * i + 1] + b[2 * i + 1];
      if (EPI == EPI_BIAS_SILU) {
        pp[i] = __floats2bfloat162_rn(x0, x1);
        x0 = silu(x0);
        x1 = silu(x1);
      }
      ph[i] = __floats2bfloat162_rn(x0, x1);
    }
  }
}

// One epilogue warp's share of a 128-row accumulator: its 32 TMEM lanes starting at t_row
// (output rows store_row ... store_row + 31; this lane's row is `row`), accumulator
// columns [col_lo, col_lo + COLS) of the tile that starts at output column n0, 64 at a
// time.  Adds the bias, applies the activation and writes bf16: through the warp's 4 KB
// staging box and one TMA store per 64 columns when use_tma (all 32 rows in the group,
// the columns in range, no pre-activation output), else with 16-byte stores per row,
// skipping a row past the group's end (valid false) and columns past N.  The 64 columns
// and their biases are loaded and converted before the warp waits for its previous
// store to have read the staging box, so that read overlaps the arithmetic.
template <int EPI, int COLS>
__device__ __forceinline__ void rows_epilogue_slab(uint32_t t_row, int col_lo, bool use_tma,
                                                   int64_t row, bool valid, int n0, int N,
                                                   const __nv_bfloat16* bias,
                                                   __nv_bfloat16* out, void* pre_out,
                                                   uint8_t* stg, const CUtensorMap* tmO,
                                                   int store_row, int lane) {
  static_assert(COLS % 64 == 0, "64-column pieces");
#pragma unroll 1
  for (int col = col_lo; col < col_lo + COLS; col += 64) {
    float v0[32], v1[32];
    if (use_tma) {
      // use_tma: every column of the piece is in range.
      uint4 bv[2][4];
      if (bias) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
          bv[i / 4][i % 4] = __ldg(reinterpret_cast<const uint4*>(bias + col + 8 * i));
      }
      uint4 packed[2][4], pre[4];
      tmem_ld_32cols(t_row + col, v0);
      tmem_ld_32cols(t_row + col + 32, v1);
      tc_wait_ld();
      bias_act_32<EPI>(v0, bv[0], bias != nullptr, packed[0], pre);
      bias_act_32<EPI>(v1, bv[1], bias != nullptr, packed[1], pre);
      if (lane == 0) bulk_wait_group_read0();
      __syncwarp();
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int chunk = i ^ (lane & 7);
        *reinterpret_cast<uint4*>(stg + lane * 128 + chunk * 16) = packed[i / 4][i % 4];
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store_2d(tmO, smem_u32(stg), n0 + col, store_row);
        bulk_commit_group();
      }
      continue;
    }
    // Rows or columns at an edge (or a pre-activation output): 16-byte stores per row.
    auto direct = [&](const float (&v)[32], int c0) {
      if (!valid || n0 + c0 >= N) return;
      const bool full32 = n0 + c0 + 32 <= N;
      uint4 b32[4];
      if (bias && full32) {
#pragma unroll
        for (int q = 0; q < 4; ++q) b32[q] = __ldg(reinterpret_cast<const uint4*>(bias + c0 + 8 * q));
      } else {
        // Columns past N: biases of the columns in range, zeros beyond.
        __nv_bfloat16* bh = reinterpret_cast<__nv_bfloat16*>(b32);
#pragma unroll
        for (int i = 0; i < 32; ++i)
          bh[i] = (bias && n0 + c0 + i < N) ? bias[c0 + i] : __float2bfloat16(0.f);
      }
      uint4 packed[4], pre[4];
      bias_act_32<EPI>(v, b32, bias != nullptr, packed, pre);
      __nv_bfloat16* o = out + row * N + n0 + c0;
      __nv_bfloat16* op = (EPI == EPI_BIAS_SILU && pre_out)
                              ? static_cast<__nv_bfloat16*>(pre_out) + (o - out)
                              : nullptr;
      if (full32) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          *reinterpret_cast<uint4*>(o + 8 * q) = packed[q];
          if (op) *reinterpret_cast<uint4*>(op + 8 * q) = pre[q];
        }
      } else {
        const __nv_bfloat16* pv = reinterpret_cast<const __nv_bfloat16*>(packed);
        const __nv_bfloat16* pr = reinterpret_cast<const __nv_bfloat16*>(pre);
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (n0 + c0 + i < N) {
            o[i] = pv[i];
            if (op) op[i] = pr[i];
          }
      }
    };
    __syncwarp();  // the TMEM loads are warp-collective
    tmem_ld_32cols(t_row + col, v0);
    tc_wait_ld();
    direct(v0, col);
    __syncwarp();
    tmem_ld_32cols(t_row + col + 32, v1);
    tc_wait_ld();
    direct(v1, col + 32);
  }
}

// ------------------------------------------------------------- expert FFN, row tiles
// A = token block [128 x 64] of the row buffer (2-D map); B = weight block [BN x 64]
// of W[g] (3-D map over [G, N, K]); D[128 x BN] in TMEM, lane = token row, column =
// output feature.  Used for large expert groups (hundreds of rows and more), where a
// 128-row tile is mostly full.  The epilogue writes each row's 32-column pieces as
// 16-byte stores; rows past the group's end belong to the next expert and are not
// written.  Eight epilogue warps: shortening the drain of one accumulator measured
// 2.7% faster on the 8-expert prefill layer than four.  A warp whose 32 rows all belong
// to the group (every warp but those of a group's last, partial row tile) stages each
// 32 x 64 piece of its output in shared memory (128-byte swizzled, 4 KB per warp) and
// writes it with one TMA store: whole 128-byte lines instead of 16-byte pieces of 32
// rows per store instruction (1.2-1.4% faster on the prefill and 256-expert layers).
// When the pre-activation is also requested, every warp stores directly.
template <int BN, int STAGES, int EPI, bool GATHER>
__global__ void __launch_bounds__(ROWS_THREADS, 1)
    tc_rows_ffn_kernel(const __grid_constant__ CUtensorMap tmX,
                       const __grid_constant__ CUtensorMap tmW,
                       const __grid_constant__ CUtensorMap tmO, const GemmArgs p) {
  static_assert(BN % 32 == 0 && BN <= 256 && (BN & (BN - 1)) == 0, "BN: power of two, <= 256");
  static_assert(EPI == EPI_BIAS_SILU || EPI == EPI_BIAS, "expert epilogues only");
  constexpr uint32_t kTmemCols = 2 * BN;
  constexpr uint32_t kIdesc = bf16_idesc(TILE_M, BN);
  constexpr uint32_t kStageBytes = (TILE_M + BN) * TC_BK * 2;
  using Smem = PipeSmem<TILE_M * TC_BK * 2, BN * TC_BK * 2, STAGES>;
  Smem& S = smem_aligned<Smem>();
  // Gathered token rows: the current tile's token ids, in the padding between the
  // pipeline state and the 1 KB-aligned epilogue staging boxes (the dynamic shared memory
  // is already at the per-block maximum, so there is no room for a static array).
  static_assert(((sizeof(Smem) + 1023) & ~size_t{1023}) - sizeof(Smem) >= TILE_M * sizeof(int) + 16,
                "room for the token ids before the staging boxes");
  int* s_tok = reinterpret_cast<int*>(
      (reinterpret_cast<uintptr_t>(&S) + sizeof(Smem) + 15) & ~static_cast<uintptr_t>(15));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.G;
  pipe_prologue<Smem, STAGES>(S, kTmemCols, p, G, TILE_M, &tmX, &tmW, 32 * ROWS_EPI_WARPS);

  const int NB = (p.N + BN - 1) / BN;
  const int total = S.pref[G] * NB;
  const int KB = (p.K + TC_BK - 1) / TC_BK;
  volatile int* abort = &S.abort;

  struct Coord {
    int g, n0, kb0, kb1;
    uint32_t bytes;
    int64_t row0, row_end;
  };
  auto decode = [&](int tile) {
    Coord c;
    c.g = find_group(S.pref, G, NB, tile);
    const int mt = S.pref[c.g + 1] - S.pref[c.g];
    const int local = tile - S.pref[c.g] * NB;
    c.n0 = (local / mt) * BN;
    c.row0 = p.offsets[c.g] + static_cast<int64_t>(local % mt) * TILE_M;
    c.row_end = p.offsets[c.g + 1];
    c.bytes = kStageBytes;
    c.kb0 = 0;
    c.kb1 = KB;
    return c;
  };

  if (warp == 0) {
    if constexpr (GATHER) {
      // Token rows straight from x: the tile's token ids are fetched by the whole warp
      // (rows past the group's end repeat its last token; an id outside [0, rows) is
      // flagged and read as token 0), then the 128-row token tile as 32 gathers of four.
      run_producer_warp<STAGES>(
          S, static_cast<int>(blockIdx.x), static_cast<int>(gridDim.x), total, decode,
          [&](const Coord& c, int ln) {
            for (int i = ln; i < TILE_M; i += 32) {
              const int64_t r = c.row0 + i < c.row_end ? c.row0 + i : c.row_end - 1;
              int t = p.gather_rows[r];
              if (t < 0 || t >= p.gather_src_rows) {
                raise_flag(p.flags, MOE_DEVERR_BAD_ROW);
                t = 0;
              }
              s_tok[i] = t;
            }
          },
          [&](const Coord& c, int kb, uint32_t sa, uint32_t sb, uint32_t bar) {
            for (int j = 0; j < TILE_M; j += 4)
              tma_gather4(sa + j * TC_BK * 2, &tmX, bar, kb * TC_BK, s_tok[j], s_tok[j + 1],
                          s_tok[j + 2], s_tok[j + 3]);
            tma_load_3d(sb, &tmW, bar, kb * TC_BK, c.n0, c.g);
          },
          abort, p.flags);
    } else if (lane == 0) {
      run_producer<STAGES>(
          S, static_cast<int>(blockIdx.x), static_cast<int>(gridDim.x), total, decode,
          [&](const Coord& c, int kb, uint32_t sa, uint32_t sb, uint32_t bar) {
            tma_load_2d(sa, &tmX, bar, kb * TC_BK, static_cast<int>(c.row0));
            tma_load_3d(sb, &tmW, bar, kb * TC_BK, c.n0, c.g);
          },
          abort, p.flags);
    }
  } else if (warp == 1) {
    if (lane == 0)
      run_mma<STAGES, BN>(S, static_cast<int>(blockIdx.x), static_cast<int>(gridDim.x), total,
                             S.tmem_base, decode, [](const Coord&) { return kIdesc; }, abort,
                             p.flags);
  } else {
    const int quad = warp & 3;  // TMEM lanes this warp may read: 32*quad .. 32*quad+31
    constexpr int kColsPerWarp = BN * 4 / ROWS_EPI_WARPS;
    const int col_lo = ((warp - 2) / 4) * kColsPerWarp;  // this warp's share of the columns
    const __nv_bfloat16* bias_base = static_cast<const __nv_bfloat16*>(p.bias);
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out);
    uint8_t* stg = reinterpret_cast<uint8_t*>(&S) + ((sizeof(Smem) + 1023) & ~size_t{1023}) +
                   (warp - 2) * 4096;
    int acc = 0;
    uint32_t aph = 0;
    for (int tile = static_cast<int>(blockIdx.x); tile < total; tile += static_cast<int>(gridDim.x)) {
      const Coord c = decode(tile);
      const bool got = mbar_wait_bounded(smem_u32(&S.tfull[acc]), aph, abort, p.flags);
      if (!__all_sync(0xffffffffu, got)) break;  // the warp-collective loads need every lane
      tc_fence_after();
      const bool use_tma = p.pre_out == nullptr && c.row0 + quad * 32 + 32 <= c.row_end &&
                           c.n0 + col_lo + kColsPerWarp <= p.N;
      const int64_t row = c.row0 + quad * 32 + lane;
      const bool valid = row < c.row_end;
      const uint32_t t_row = S.tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                             static_cast<uint32_t>(acc * BN);
      const __nv_bfloat16* bias =
          bias_base ? bias_base + static_cast<int64_t>(c.g) * p.N + c.n0 : nullptr;
      rows_epilogue_slab<EPI, kColsPerWarp>(t_row, col_lo, use_tma, row, valid, c.n0, p.N, bias,
                                           out, p.pre_out, stg, &tmO,
                                           static_cast<int>(c.row0) + quad * 32, lane);
      tc_fence_before();
      mbar_arrive(smem_u32(&S.tempty[acc]));
      acc ^= 1;
      if (acc == 0) aph ^= 1u;
    }
    if (lane == 0) bulk_wait_group0();
  }
  pipe_teardown(S, kTmemCols);
}

// ------------------------------------------------------------- router GEMM
// A = token block [128 x 64] of x; B = expert block [BN x 64] of W_g; D[128 x BN],
// lane = token, column = expert.  When there are too few tiles to fill the GPU the
// K dimension is split across CTAs: split s writes its partial sums to
// out + s * split_stride, and the softmax/top-k kernel adds the splits in order and
// the logit bias (so every logit is one fixed-order fp32 sum).
template <int BN, int STAGES>
__global__ void __launch_bounds__(TC_THREADS, 1)
    tc_router_kernel(const __grid_constant__ CUtensorMap tmX,
                     const __grid_constant__ CUtensorMap tmW, const GemmArgs p) {
  static_assert(BN >= 16 && BN <= 256 && (BN & (BN - 1)) == 0, "BN: power of two in [16, 256]");
  constexpr uint32_t kTmemCols = (2 * BN < 32) ? 32 : 2 * BN;
  constexpr uint32_t kIdesc = bf16_idesc(TILE_M, BN);
  constexpr uint32_t kStageBytes = (TILE_M + BN) * TC_BK * 2;
  constexpr int CH = BN < 32 ? BN : 32;
  using Smem = PipeSmem<TILE_M * TC_BK * 2, BN * TC_BK * 2, STAGES>;
  Smem& S = smem_aligned<Smem>();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pipe_prologue<Smem, STAGES>(S, kTmemCols, p, 1, TILE_M, &tmX, &tmW);

  const int NB = (p.N + BN - 1) / BN;
  const int MT = S.pref[1];
  const int KB = (p.K + TC_BK - 1) / TC_BK;
  const int splits = p.ksplit > 1 ? p.ksplit : 1;
  const int kb_per = (KB + splits - 1) / splits;
  const int total = MT * NB * splits;
  volatile int* abort = &S.abort;

  struct Coord {
    int n0, split, kb0, kb1;
    uint32_t bytes;
    int64_t row0;
  };
  auto decode = [&](int tile) {
    Coord c;
    c.bytes = kStageBytes;
    c.split = tile / (MT * NB);
    const int rem = tile % (MT * NB);
    c.n0 = (rem / MT) * BN;
    c.row0 = static_cast<int64_t>(rem % MT) * TILE_M;
    c.kb0 = c.split * kb_per;
    c.kb1 = c.kb0 + kb_per < KB ? c.kb0 + kb_per : KB;
    return c;
  };

  if (warp == 0) {
    if (lane == 0)
      run_producer<STAGES>(
          S, static_cast<int>(blockIdx.x), static_cast<int>(gridDim.x), total, decode,
          [&](const Coord& c, int kb, uint32_t sa, uint32_t sb, uint32_t bar) {
            tma_load_2d(sa, &tmX, bar, kb * TC_BK, static_cast<int>(c.row0));
            tma_load_3d(sb, &tmW, bar, kb * TC_BK, c.n0, 0);
          },
          abort, p.flags);
  } else if (warp == 1) {
    if (lane == 0)
      run_mma<STAGES, BN>(S, static_cast<int>(blockIdx.x), static_cast<int>(gridDim.x), total,
                             S.tmem_base, decode, [](const Coord&) { return kIdesc; }, abort,
                             p.flags);
  } else {
    const int quad = warp & 3;
    int acc = 0;
    uint32_t aph = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
      const Coord c = decode(tile);
      float* out = static_cast<float*>(p.out) + static_cast<int64_t>(c.split) * p.split_stride;
      const bool got = mbar_wait_bounded(smem_u32(&S.tfull[acc]), aph, abort, p.flags);
      if (!__all_sync(0xffffffffu, got)) break;
      tc_fence_after();
      const int64_t row = c.row0 + quad * 32 + lane;
      const uint32_t t_row = S.tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                             static_cast<uint32_t>(acc * BN);
#pragma unroll 1
      for (int col = 0; col < BN; col += CH) {
        float v[CH];
        if constexpr (CH == 32)
          tmem_ld_32cols(t_row + col, v);
        else
          tmem_ld_16cols(t_row + col, v);
        tc_wait_ld();
        if (row < p.m_rows) {
          const int e0 = c.n0 + col;
          float* dst = out + row * p.N + e0;
          if ((p.N & 3) == 0 && e0 + CH <= p.N) {
            // Whole chunk in range and 16-byte aligned (N % 4 == 0, e0 % 16 == 0).
#pragma unroll
            for (int i = 0; i < CH; i += 4)
              *reinterpret_cast<float4*>(dst + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
          } else {
#pragma unroll
            for (int i = 0; i < CH; ++i)
              if (e0 + i < p.N) dst[i] = v[i];
          }
        }
      }
      tc_fence_before();
      mbar_arrive(smem_u32(&S.tempty[acc]));
      acc ^= 1;
      if (acc == 0) aph ^= 1u;
    }
  }
  pipe_teardown(S, kTmemCols);
}

// Expert GEMM on 256-row token tiles (groups larger than 128 rows).  A k-block stage holds
// the tile's two 128-row token halves and one 256-row block of the weights, and the MMA
// thread issues both halves against the shared weight block into two accumulators (TMEM
// columns 0-255 and 256-511): 64 KB of operands per 2 x (128 x 256 x 64) MMAs, where two
// 128-row tiles need 96 KB, so the same shared-memory ring (three 64 KB stages instead of
// four of 48 KB) carries a third more MMA work per byte -- the main loop of the 128-row
// kernel waits on operand delivery, not on the tensor core.  With all 512 columns in use
// the accumulators are not double-buffered: the epilogue drains the first half and
// releases it before the second, so the next tile's first-half MMAs start during the
// second half's drain while the producer refills the ring.  A tile with at most 128 rows
// left (a group's tail) loads and computes only its first half.
template <int STAGES, int EPI, int EPI_WARPS, bool STAGED>
__global__ void __launch_bounds__(64 + 32 * EPI_WARPS, 1)
    tc_rows_wide_ffn_kernel(const __grid_constant__ CUtensorMap tmX,
                            const __grid_constant__ CUtensorMap tmW,
                            const __grid_constant__ CUtensorMap tmO, const GemmArgs p) {
  static_assert(EPI == EPI_BIAS_SILU || EPI == EPI_BIAS, "expert epilogues only");
  static_assert(EPI_WARPS % 4 == 0 && EPI_WARPS >= 4 && EPI_WARPS <= 16, "whole lane quadrants");
  constexpr int BN = 256;
  constexpr int TM = 2 * TILE_M;
  constexpr uint32_t kTmemCols = 2 * BN;
  constexpr uint32_t kIdesc = bf16_idesc(TILE_M, BN);
  constexpr uint32_t kHalfBytes = TILE_M * TC_BK * 2;
  constexpr uint32_t kWeightBytes = BN * TC_BK * 2;
  using Smem = PipeSmem<2 * kHalfBytes, kWeightBytes, STAGES>;
  Smem& S = smem_aligned<Smem>();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.G;
  pipe_prologue<Smem, STAGES>(S, kTmemCols, p, G, TM, &tmX, &tmW, 32 * EPI_WARPS);

  const int NB = (p.N + BN - 1) / BN;
  const int total = S.pref[G] * NB;
  const int KB = (p.K + TC_BK - 1) / TC_BK;
  volatile int* abort = &S.abort;

  struct Coord {
    int g, n0, kb0, kb1;
    bool two;  // the second 128-row half holds rows of the group
    uint32_t bytes;
    int64_t row0, row_end;
  };
  auto decode = [&](int tile) {
    Coord c;
    c.g = find_group(S.pref, G, NB, tile);
    const int mt = S.pref[c.g + 1] - S.pref[c.g];
    const int local = tile - S.pref[c.g] * NB;
    c.n0 = (local / mt) * BN;
    c.row0 = p.offsets[c.g] + static_cast<int64_t>(local % mt) * TM;
    c.row_end = p.offsets[c.g + 1];
    c.two = c.row_end - c.row0 > TILE_M;
    c.bytes = kWeightBytes + (c.two ? 2u : 1u) * kHalfBytes;
    c.kb0 = 0;
    c.kb1 = KB;
    return c;
  };
  const int first = static_cast<int>(blockIdx.x), step = static_cast<int>(gridDim.x);

  if (warp == 0) {
    if (lane == 0)
      run_producer<STAGES>(
          S, first, step, total, decode,
          [&](const Coord& c, int kb, uint32_t sa, uint32_t sb, uint32_t bar) {
            tma_load_2d(sa, &tmX, bar, kb * TC_BK, static_cast<int>(c.row0));
            if (c.two)
              tma_load_2d(sa + kHalfBytes, &tmX, bar, kb * TC_BK, static_cast<int>(c.row0) + TILE_M);
            tma_load_3d(sb, &tmW, bar, kb * TC_BK, c.n0, c.g);
          },
          abort, p.flags);
  } else if (warp == 1) {
    if (lane == 0) {
      // tempty[h]: the epilogue has drained accumulator half h of the previous tile (it
      // arrives on both once per tile, also for a one-half tile); tfull[0]: the tile's MMAs
      // are complete.
      int s = 0;
      uint32_t ph = 0, aph = 0;
      bool ok = true, issued_any = false;
      for (int tile = first; ok && tile < total; tile += step) {
        const Coord c = decode(tile);
        if (!mbar_wait_bounded(smem_u32(&S.tempty[0]), aph ^ 1u, abort, p.flags)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int kb = c.kb0; kb < c.kb1; ++kb) {
          if (!mbar_wait_bounded(smem_u32(&S.full[s]), ph, abort, p.flags)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(S.a[s]), b0 = smem_u32(S.b[s]);
#pragma unroll
          for (int kk = 0; kk < TC_BK / 16; ++kk)
            tc_mma_bf16(S.tmem_base, sw128_kmajor_desc(a0 + kk * 32),
                        sw128_kmajor_desc(b0 + kk * 32), kIdesc,
                        (kb != c.kb0 || kk != 0) ? 1u : 0u);
          issued_any = true;
          if (c.two) {
            if (kb == c.kb0) {
              if (!mbar_wait_bounded(smem_u32(&S.tempty[1]), aph ^ 1u, abort, p.flags)) {
                ok = false;
                break;
              }
              tc_fence_after();
            }
#pragma unroll
            for (int kk = 0; kk < TC_BK / 16; ++kk)
              tc_mma_bf16(S.tmem_base + BN, sw128_kmajor_desc(a0 + kHalfBytes + kk * 32),
                          sw128_kmajor_desc(b0 + kk * 32), kIdesc,
                          (kb != c.kb0 || kk != 0) ? 1u : 0u);
          }
          tc_commit(smem_u32(&S.empty[s]));
          if (++s == STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(smem_u32(&S.tfull[0]));
        aph ^= 1u;
      }
      // Unwinding: every MMA issued by this thread completes before TMEM is released.
      if (!ok && issued_any) {
        tc_commit(smem_u32(&S.drain));
        mbar_wait_unwind(smem_u32(&S.drain), 0);
      }
    }
  } else {
    const int quad = warp & 3;  // TMEM lanes this warp may read: 32*quad .. 32*quad+31
    constexpr int kColsPerWarp = BN * 4 / EPI_WARPS;
    const int col_lo = ((warp - 2) / 4) * kColsPerWarp;  // this warp's share of the columns
    const __nv_bfloat16* bias_base = static_cast<const __nv_bfloat16*>(p.bias);
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out);
    uint8_t* stg = reinterpret_cast<uint8_t*>(&S) + ((sizeof(Smem) + 1023) & ~size_t{1023}) +
                   (warp - 2) * 4096;
    uint32_t aph = 0;
    for (int tile = first; tile < total; tile += step) {
      const Coord c = decode(tile);
      const bool got = mbar_wait_bounded(smem_u32(&S.tfull[0]), aph, abort, p.flags);
      if (!__all_sync(0xffffffffu, got)) break;  // the warp-collective loads need every lane
      tc_fence_after();
      const __nv_bfloat16* bias =
          bias_base ? bias_base + static_cast<int64_t>(c.g) * p.N + c.n0 : nullptr;
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        if (h == 0 || c.two) {
          const int64_t r0 = c.row0 + h * TILE_M + quad * 32;
          const bool use_tma =
              STAGED && p.pre_out == nullptr && r0 + 32 <= c.row_end &&
              c.n0 + col_lo + kColsPerWarp <= p.N;
          const uint32_t t_row =
              S.tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + static_cast<uint32_t>(h * BN);
          rows_epilogue_slab<EPI, kColsPerWarp>(t_row, col_lo, use_tma, r0 + lane,
                                                r0 + lane < c.row_end, c.n0, p.N, bias, out,
                                                p.pre_out, stg, &tmO, static_cast<int>(r0), lane);
        }
        tc_fence_before();
        mbar_arrive(smem_u32(&S.tempty[h]));
      }
      aph ^= 1u;
    }
    if (lane == 0) bulk_wait_group0();
  }
  pipe_teardown(S, kTmemCols);
}

template <int TB, int STAGES, int EPI>
cudaError_t launch_ffn(const GemmArgs& a, int sm_count, cudaStream_t stream) {
  if (!a.sk_ctr || !a.sk_part) return cudaErrorInvalidValue;
  CUtensorMap tmW, tmX;
  // Token rows: 32-row boxes of the expert-ordered rows, or one-row boxes of x to gather.
  const bool ok_x = a.gather_rows ? rows_map(&tmX, a.gather_src, a.gather_src_rows, a.K, 1)
                                  : rows_map(&tmX, a.A, a.rows_alloc, a.K, tok_box(TB));
  if (!stacked_map(&tmW, a.B, a.G, a.N, a.K, TILE_M) || !ok_x) return cudaErrorInvalidValue;
  using Smem = PipeSmem<TILE_M * TC_BK * 2, TB * TC_BK * 2, STAGES>;
  // One CTA per SM; the parked pieces and counters are sized for kMaxSmsForSizing.
  const int grid = std::min(sm_count, kMaxSmsForSizing);
  const size_t smem = sizeof(Smem) + 1024;
  const size_t smem_gather = smem + TB * sizeof(int) + 16;
  if constexpr (EPI == EPI_BIAS_SILU) {
    if (a.gather_rows && a.comb_out)
      return launch_pipe(tc_ffn_kernel<TB, STAGES, EPI, true, true>, smem_gather, grid, tmW, tmX,
                         a, stream);
    if (a.gather_rows)
      return launch_pipe(tc_ffn_kernel<TB, STAGES, EPI, true, false>, smem_gather, grid, tmW,
                         tmX, a, stream);
  }
  if (a.comb_out)
    return launch_pipe(tc_ffn_kernel<TB, STAGES, EPI, false, true>, smem, grid, tmW, tmX, a,
                       stream);
  if (a.gather_rows) return cudaErrorInvalidValue;
  return launch_pipe(tc_ffn_kernel<TB, STAGES, EPI, false, false>, sizeof(Smem) + 1024, grid,
                     tmW, tmX, a, stream);
}

template <int BN, int STAGES, int EPI>
cudaError_t launch_rows_ffn(const GemmArgs& a, int sm_count, cudaStream_t stream) {
  CUtensorMap tmX, tmW;
  // Token rows: 128-row boxes of the expert-ordered rows, or one-row boxes of x to gather.
  const bool ok_x = a.gather_rows ? rows_map(&tmX, a.gather_src, a.gather_src_rows, a.K, 1)
                                  : rows_map(&tmX, a.A, a.rows_alloc, a.K, TILE_M);
  if (!ok_x || !stacked_map(&tmW, a.B, a.G, a.N, a.K, BN)) return cudaErrorInvalidValue;
  // Upper bound on tiles: sum_g ceil(rows_g / 128) <= rows_alloc / 128 + G.
  const int64_t bound = ((a.rows_alloc + TILE_M - 1) / TILE_M + a.G) * ((a.N + BN - 1) / BN);
  const int grid = static_cast<int>(std::min<int64_t>(bound, sm_count));
  using Smem = PipeSmem<TILE_M * TC_BK * 2, BN * TC_BK * 2, STAGES>;
  CUtensorMap tmO;
  if (!rows_map(&tmO, a.out, a.rows_alloc, a.N, 32)) return cudaErrorInvalidValue;
  const size_t smem = ((sizeof(Smem) + 1023) & ~size_t{1023}) + 8 * 4096 + 1024;
  auto go = [&](auto kern) -> cudaError_t {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    if (grid <= 0) return cudaSuccess;
    launch_pdl(kern, grid, ROWS_THREADS, smem, stream, tmX, tmW, tmO, a);
    return cudaGetLastError();
  };
  if constexpr (EPI == EPI_BIAS_SILU) {
    if (a.gather_rows) return go(tc_rows_ffn_kernel<BN, STAGES, EPI, true>);
  }
  if (a.gather_rows) return cudaErrorInvalidValue;
  return go(tc_rows_ffn_kernel<BN, STAGES, EPI, false>);
}

template <int STAGES, int EPI, int EPI_WARPS = ROWS_EPI_WARPS, bool STAGED = true>
cudaError_t launch_rows_wide_ffn(const GemmArgs& a, int sm_count, cudaStream_t stream) {
  constexpr int BN = 256, TM = 2 * TILE_M;
  CUtensorMap tmX, tmW, tmO;
  if (!rows_map(&tmX, a.A, a.rows_alloc, a.K, TILE_M) ||
      !stacked_map(&tmW, a.B, a.G, a.N, a.K, BN) || !rows_map(&tmO, a.out, a.rows_alloc, a.N, 32))
    return cudaErrorInvalidValue;
  // Upper bound on tiles: sum_g ceil(rows_g / 256) <= rows_alloc / 256 + G.
  const int64_t bound = ((a.rows_alloc + TM - 1) / TM + a.G) * ((a.N + BN - 1) / BN);
  const int grid = static_cast<int>(std::min<int64_t>(bound, sm_count));
  using Smem = PipeSmem<2 * TILE_M * TC_BK * 2, BN * TC_BK * 2, STAGES>;
  const size_t smem =
      ((sizeof(Smem) + 1023) & ~size_t{1023}) + (STAGED ? EPI_WARPS * 4096 : 0) + 1024;
  auto kern = tc_rows_wide_ffn_kernel<STAGES, EPI, EPI_WARPS, STAGED>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  if (grid <= 0) return cudaSuccess;
  launch_pdl(kern, grid, 64 + 32 * EPI_WARPS, smem, stream, tmX, tmW, tmO, a);
  return cudaGetLastError();
}

template <int BN, int STAGES>
cudaError_t launch_router(const GemmArgs& a, int sm_count, cudaStream_t stream) {
  CUtensorMap tmX, tmW;
  if (!rows_map(&tmX, a.A, a.m_rows, a.K, TILE_M) || !stacked_map(&tmW, a.B, 1, a.N, a.K, BN))
    return cudaErrorInvalidValue;
  const int64_t bound = ((a.m_rows + TILE_M - 1) / TILE_M) * ((a.N + BN - 1) / BN) *
                        (a.ksplit > 1 ? a.ksplit : 1);
  const int grid = static_cast<int>(std::min<int64_t>(bound, sm_count));
  using Smem = PipeSmem<TILE_M * TC_BK * 2, BN * TC_BK * 2, STAGES>;
  return launch_pipe(tc_router_kernel<BN, STAGES>, sizeof(Smem) + 1024, grid, tmX, tmW, a, stream);
}

// Token-block height for a weights-as-M expert GEMM: the smallest power of two
// (32..128) that holds the largest group the routing can produce.
template <int EPI>
cudaError_t launch_ffn_for(const GemmArgs& a, int max_group, int sm_count, cudaStream_t stream) {
  if (max_group <= 32) return launch_ffn<32, 11, EPI>(a, sm_count, stream);
  if (max_group <= 64) return launch_ffn<64, 9, EPI>(a, sm_count, stream);
  return launch_ffn<128, 7, EPI>(a, sm_count, stream);
}

// kSmallGroup (kernels.h) bounds the groups of the weights-as-M kernel: there a
// 128-row tile would be mostly padding, while 128 weight rows always fill the MMA's M
// side.  Larger groups use row tiles, whose main loop measured faster.

// Router tile width for E experts: the narrowest power of two that covers them, at
// most 128.
int router_bn(int E) { return E <= 16 ? 16 : E <= 32 ? 32 : E <= 64 ? 64 : 128; }

}  // namespace

int router_splits(int64_t T, int E, int d, int sms) {
  const int64_t tiles = ((T + TILE_M - 1) / TILE_M) * ((E + router_bn(E) - 1) / router_bn(E));
  const int64_t kb = (d + TC_BK - 1) / TC_BK;
  const int64_t by_fill = tiles > 0 ? sms / tiles : 1;
  const int64_t s = std::max<int64_t>(1, std::min<int64_t>(by_fill, kb / 4));
  // The same number of k-blocks per split as the kernel uses; no empty split.
  const int64_t per = (kb + s - 1) / s;
  return static_cast<int>((kb + per - 1) / per);
}

// Groups larger than 128 rows.  256-row tiles carry a third more MMA work per operand
// byte, which pays where each expert's weight blocks are reused by many row tiles (512 or
// more rows per expert on average): there the tensor core bounds the main loop, and the
// 256-row tiles run it about 1.4x faster per FLOP.  With fewer rows per expert the weight
// stream from DRAM bounds both tile shapes, while the 256-row tiles pay for their
// epilogue (their accumulators fill TMEM, so it does not overlap the next tile's MMAs) and
// for half-empty last tiles.  Gathered token rows and a pre-activation output keep the
// 128-row tiles (their epilogue stores row by row, which the wide tile would expose).
constexpr int64_t kWideMinRowsPerGroup = 512;

template <int EPI>
cudaError_t launch_rows_for(const GemmArgs& a, int sm_count, cudaStream_t stream) {
  const bool wide = a.gather_rows == nullptr && a.pre_out == nullptr &&
                    a.rows_alloc >= kWideMinRowsPerGroup * a.G;
  return wide ? launch_rows_wide_ffn<3, EPI>(a, sm_count, stream)
              : launch_rows_ffn<256, 4, EPI>(a, sm_count, stream);
}


cudaError_t launch_tc_gemm_bf16(const GemmArgs& a, int epi, int sm_count, cudaStream_t stream) {
  // Gathered token rows exist for the first expert GEMM only, the fused top-1 combine for
  // the second on the weights-as-M kernel only.
  if (a.gather_rows && (epi != EPI_BIAS_SILU || !a.gather_src || a.gather_src_rows < 1))
    return cudaErrorInvalidValue;
  if (a.comb_out &&
      (a.max_group > kSmallGroup || a.comb_rows < 1 || a.comb_cols < 8 || a.comb_cols % 8 ||
       (epi == EPI_BIAS ? !a.comb_token || !a.comb_w : epi == EPI_BIAS_SILU ? !a.comb_slot : true)))
    return cudaErrorInvalidValue;
  switch (epi) {
    case EPI_BIAS_SILU:
      return a.max_group > kSmallGroup ? launch_rows_for<EPI_BIAS_SILU>(a, sm_count, stream)
                                       : launch_ffn_for<EPI_BIAS_SILU>(a, a.max_group, sm_count, stream);
    case EPI_BIAS:
      return a.max_group > kSmallGroup ? launch_rows_for<EPI_BIAS>(a, sm_count, stream)
                                       : launch_ffn_for<EPI_BIAS>(a, a.max_group, sm_count, stream);
    default:
      switch (router_bn(a.N)) {
        case 16: return launch_router<16, 8>(a, sm_count, stream);
        case 32: return launch_router<32, 8>(a, sm_count, stream);
        case 64: return launch_router<64, 8>(a, sm_count, stream);
        default: return launch_router<128, 6>(a, sm_count, stream);
      }
  }
}

}  // namespace moe
