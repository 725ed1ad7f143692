// Tensor-core GEMM engine for sm_103a: tcgen05.mma with fp32 accumulators in
// TMEM, operands staged in shared memory by TMA (128-byte swizzle), persistent
// CTAs, one elected thread issuing the MMAs.
//
// One launch computes a list of "groups"; each group is an output matrix
//     D (M x N) = sum over its segments s of A_s B_s^T
// followed by a fused epilogue.  The segments of a group are the shards of a
// tensor-parallel reduction: the row-parallel linear's forward sum over shards
// (g operator) and the column-parallel linear's backward sum (f operator) run
// as one fp32 accumulation in TMEM in fixed shard order, so the per-shard
// partial products never reach HBM ("Megatron" walkthrough, sections
// ColumnParallelLinear and RowParallelLinear; "Megatron tensor / model
// parallelism" notes, section MLP层的通讯量分析).
//
// CTA layout (576 threads):
//   warp 0       tile scheduler + TMA producer (one lane)
//   warp 1       TMEM allocator + MMA issuer (one lane)
//   warps 2..17  epilogue: TMEM -> registers -> fused op -> global; four warps
//                per TMEM lane quarter, each taking a quarter of the tile's
//                columns (enough warps per SM sub-partition to hide the
//                latency of the GELU / GELU' arithmetic and the stores)
// Tile 128 x 256 x 64, 4-stage smem ring, two TMEM accumulators (2 x 256
// columns) so the epilogue of one tile overlaps the main loop of the next.
// Tiles are handed out dynamically: each CTA starts with tile blockIdx.x and
// then takes the next unclaimed tile from a global counter, so launches that
// mix long-K and short-K outputs (listed longest first) balance across SMs.
// The producer passes each tile id to the MMA and epilogue warps through a
// small shared-memory ring.
// Every wait is bounded: after the limit the thread records a timeout in the
// device error word, raises a CTA-wide abort flag and the CTA winds down
// (in-flight copies and MMAs drained, TMEM freed) instead of hanging.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "tp_device.cuh"
#include "tp_internal.h"

namespace tp {
namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;
constexpr int STAGES = 4;
constexpr int A_TILE_BYTES = BM * BK * 2;  // 16 KB
constexpr int B_TILE_BYTES = BN * BK * 2;  // 32 KB
constexpr int STAGE_BYTES = A_TILE_BYTES + B_TILE_BYTES;
constexpr int TMEM_COLS = 2 * BN;  // two fp32 accumulators
constexpr int NUM_EPI_WARPS = kEpiWarps;  // four per TMEM lane quarter, each a quarter of the columns
constexpr int EPI_PARTS = NUM_EPI_WARPS / 4;  // column parts of a tile
constexpr int NUM_THREADS = 64 + 32 * NUM_EPI_WARPS;
constexpr int TILE_RING = 4;      // tile ids handed from the producer to the other roles
constexpr int MN_BOX_BYTES = 64 * BK * 2;  // one 64(MN) x 64(K) box: 8 KB
constexpr int BAR_BYTES = 512;
constexpr int EPI_STAGE_BYTES = 32 * 64;  // per epilogue warp: 32 rows x 64 bytes
constexpr int EPI_WARP_BYTES = EPI_STAGE_BYTES;
// Per-group tile table in shared memory (the producer's decode reads it
// instead of the kernel parameters, whose dynamically indexed loads miss the
// constant cache).
struct GrpLite {
  int tile_begin, tiles_m, tiles_n;
  int flags;  // bit 0: causal tiles only (tri); bit 1: column tiles fastest; bit 2: striped;
              // bits 8..15: kr_mode; bits 16..23: groups in the stripe; bits 24..31: its first group
};
constexpr int TBL_BYTES = 1024;
static_assert(kMaxGroups * sizeof(GrpLite) <= TBL_BYTES, "group table does not fit");
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + BAR_BYTES + NUM_EPI_WARPS * EPI_WARP_BYTES +
                           TBL_BYTES + 1024;  // + alignment slack

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

struct WaitCtx {
  volatile int* abort_flag;
  unsigned* err;
  unsigned long long limit_ns;
};

// Bounded wait on an mbarrier phase.  Returns false on abort or timeout.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, const WaitCtx& w) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*w.abort_flag) return false;
    if (global_ns() - t0 > w.limit_ns) {
      *w.abort_flag = 1;
      atomicOr(w.err, kErrTimeout);
      return false;
    }
  }
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, uint64_t map, uint32_t bar, int c0,
                                            int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(map), "r"(bar), "r"(c0), "r"(c1));
}

// 3D tile load: an MN-major operand viewed as (64 MN, K rows, MN / 64 blocks);
// one box brings all of a tile's 64-wide blocks, stacked 8 KB apart.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, uint64_t map, uint32_t bar, int c0,
                                            int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(map), "r"(bar), "r"(c0), "r"(c1), "r"(c2));
}

__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, uint64_t map,
                                                 uint32_t bar_cluster, int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(map), "r"(bar_cluster), "r"(c0), "r"(c1), "r"(c2));
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor (tcgen05 format): start address, leading and
// stride byte offsets (16-byte units), version 1 at bit 46, 128-byte swizzle.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;  // SWIZZLE_128B
  return d;
}

// Instruction descriptor of tcgen05.mma kind::f16: D f32, A and B bf16,
// transpose bits select MN-major operands, N >> 3 at bit 17, M >> 4 at bit 24.
__device__ __forceinline__ uint32_t idesc_bf16(int a_mn, int b_mn, int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(a_mn) << 15) |
         (static_cast<uint32_t>(b_mn) << 16) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(BM >> 4) << 24);
}

__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t* r) {
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
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ---------------------------------------------------------------------------
// Tile decode (identical sequence for all three roles)
// ---------------------------------------------------------------------------
struct TileCoord {
  int g, m0, n0;
};

template <int ROWS, bool ATTN>
__device__ __forceinline__ TileCoord decode_tile_rows(const TcGemmParams& p, const GrpLite* L, int tile) {
  if (tile < p.interleave_tiles) {
    // Leading groups share the row tiling.  They are enumerated in super-rows
    // of GM row blocks; inside a super-row, column tile by column tile (across
    // the groups) and row block fastest.  GM = 1 finishes row blocks one after
    // the other (their dependants can start early); GM = all rows streams each
    // column tile's operand once (large operands stay L2-friendly).
    const int GM = p.interleave_gm;
    const int per_super = GM * p.interleave_nt;
    const int sr = tile / per_super;
    const int m_lo = sr * GM;
    const int gm = min(GM, L[0].tiles_m - m_lo);
    const int r = tile - sr * per_super;
    int nt = r / gm;
    const int mt = m_lo + (r - nt * gm);
    int g = 0;
    while (nt >= L[g].tiles_n) {
      nt -= L[g].tiles_n;
      ++g;
    }
    TileCoord c;
    c.g = g;
    c.m0 = mt * ROWS;
    c.n0 = nt * BN;
    return c;
  }
  int g = p.interleave_groups;
  const int ng = p.num_groups;
  while (g + 1 < ng && tile >= L[g + 1].tile_begin) ++g;
  int local = tile - L[g].tile_begin;
  if (ATTN && (L[g].flags & 4)) {
    // a stripe of identical groups: consecutive tiles cycle through the
    // groups, each group's tiles in its own order (longest contraction first)
    const int first = (L[g].flags >> 24) & 0xff, n = (L[g].flags >> 16) & 0xff;
    const int t = tile - L[first].tile_begin;
    g = first + t % n;
    local = t / n;
  }
  const GrpLite G = L[g];
  TileCoord c;
  c.g = g;
  if (ATTN && (G.flags & 1)) {
    // causal: only the tiles with a column at or before their last row, row
    // block by row block (row block mt has min(tiles_n, (mt+1) ROWS / bn
    // rounded up) of them)
    int mt = 0, acc = 0;
    for (; mt < G.tiles_m - 1; ++mt) {
      const int cnt = min(G.tiles_n, (mt * ROWS + ROWS - 1) / BN + 1);
      if (local < acc + cnt) break;
      acc += cnt;
    }
    c.m0 = mt * ROWS;
    c.n0 = (local - acc) * BN;
    return c;
  }
  if (G.flags & 2) {
    // column tiles fastest: consecutive tiles share the row block of A
    c.m0 = (local / G.tiles_n) * ROWS;
    c.n0 = (local % G.tiles_n) * BN;
    return c;
  }
  const int kr = ATTN ? ((G.flags >> 8) & 0xff) : 0;
  if (ATTN && (kr == KR_END || kr == KR_BEGIN)) {
    // causal contraction ranges: a row block's column tiles together (they
    // share its A rows), longest contraction first
    int mt = local / G.tiles_n;
    if (kr == KR_END) mt = G.tiles_m - 1 - mt;
    c.m0 = mt * ROWS;
    c.n0 = (local % G.tiles_n) * BN;
    return c;
  }
  int mt = local % G.tiles_m;
  c.m0 = mt * ROWS;
  c.n0 = (local / G.tiles_m) * BN;
  return c;
}

// Fills the shared group table (all threads of the CTA may take part).
__device__ __forceinline__ void fill_group_table(const TcGemmParams& p, GrpLite* L, int tid, int nthreads) {
  for (int i = tid; i < p.num_groups; i += nthreads) {
    const GemmGroup& G = p.grp[i];
    L[i] = GrpLite{G.tile_begin, G.tiles_m, G.tiles_n,
                   (G.tri ? 1 : 0) | (G.n_fastest ? 2 : 0) | (G.stripe_n > 1 ? 4 : 0) | (G.kr_mode << 8) |
                       (G.stripe_n << 16) | (G.stripe_first << 24)};
  }
}

// k-block range [kb0, kb1) of a tile (ROWS rows from m0, columns from n0) of
// group G for a contraction of length K: everything, or the causal part.
template <int ROWS, bool ATTN>
__device__ __forceinline__ void tile_kb_range(const GemmGroup& G, int K, int m0, int n0, int& kb0,
                                              int& kb1) {
  const int nk = (K + BK - 1) / BK;
  kb0 = 0;
  kb1 = nk;
  if (!ATTN) return;
  if (G.kr_mode == KR_TRI) {
    if (n0 > m0 + ROWS - 1) kb1 = 0;
  } else if (G.kr_mode == KR_END) {
    kb1 = min(nk, (m0 + ROWS + BK - 1) / BK);
  } else if (G.kr_mode == KR_BEGIN) {
    kb0 = min(nk, m0 / BK);
  }
}

// A tile with no k-blocks: its accumulator is never written, the epilogue
// works on zeros.
template <int ROWS, bool ATTN>
__device__ __forceinline__ bool tile_empty(const TcGemmParams& p, const GemmGroup& G, int m0, int n0) {
  if (G.k_empty) return true;
  if (!ATTN || G.kr_mode == KR_NONE) return false;
  int kb0, kb1;
  tile_kb_range<ROWS, ATTN>(G, p.seg[G.seg_begin].K, m0, n0, kb0, kb1);
  return kb1 <= kb0;
}

// ---------------------------------------------------------------------------
// Epilogue of one 32-column chunk of one row
// ---------------------------------------------------------------------------
__device__ __forceinline__ void store_chunk(void* base, int out_type, int64_t ld, int row, int n,
                                            const float* v, int ncols, bool vec) {
  if (out_type == OUT_BF16) {
    __nv_bfloat16* o = static_cast<__nv_bfloat16*>(base) + static_cast<int64_t>(row) * ld + n;
    if (vec) {
      uint4* o4 = reinterpret_cast<uint4*>(o);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint4 w;
        w.x = pack_bf16x2(v[8 * q + 0], v[8 * q + 1]);
        w.y = pack_bf16x2(v[8 * q + 2], v[8 * q + 3]);
        w.z = pack_bf16x2(v[8 * q + 4], v[8 * q + 5]);
        w.w = pack_bf16x2(v[8 * q + 6], v[8 * q + 7]);
        o4[q] = w;
      }
    } else {
      _Pragma("unroll") for (int j = 0; j < 32; ++j) if (j < ncols) o[j] = __float2bfloat16_rn(v[j]);
    }
  } else {
    float* o = static_cast<float*>(base) + static_cast<int64_t>(row) * ld + n;
    if (vec) {
      float4* o4 = reinterpret_cast<float4*>(o);
#pragma unroll
      for (int q = 0; q < 8; ++q)
        o4[q] = make_float4(v[4 * q + 0], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
    } else {
      _Pragma("unroll") for (int j = 0; j < 32; ++j) if (j < ncols) o[j] = v[j];
    }
  }
}

__device__ __forceinline__ void load_bf16_chunk(const __nv_bfloat16* src, float* v, int ncols,
                                                bool vec) {
  if (vec) {
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 w = __ldg(s4 + q);
      unpack_bf16x2(w.x, v[8 * q + 0], v[8 * q + 1]);
      unpack_bf16x2(w.y, v[8 * q + 2], v[8 * q + 3]);
      unpack_bf16x2(w.z, v[8 * q + 4], v[8 * q + 5]);
      unpack_bf16x2(w.w, v[8 * q + 6], v[8 * q + 7]);
    }
  } else {
    _Pragma("unroll") for (int j = 0; j < 32; ++j) v[j] = j < ncols ? bf2f(src[j]) : 0.f;
  }
}

// ---------------------------------------------------------------------------
// Coalesced row-block transfers.  After the TMEM load, lane l of a warp holds
// row (row0 + l) of a 32 x 32 chunk.  Stores and loads of such a chunk go
// through a per-warp shared-memory stage (16-byte units, XOR-swizzled so both
// the row-per-lane side and the coalesced side are free of bank conflicts),
// so each global access instruction of the warp covers whole 64-byte (bf16)
// or 128-byte (fp32) row segments instead of 32 half-filled sectors.
// ---------------------------------------------------------------------------
// The warp's stage may still be read by its last bulk tensor store: lane 0
// waits for those reads, then the warp may write it again.
__device__ __forceinline__ void stage_acquire(int lane) {
  if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
  __syncwarp();
}
// A warp's bulk tensor load of one auxiliary chunk (the dGELU / softmax
// backward operand) into its stage: the warp's own mbarrier and its phase.
struct AuxLoad {
  uint32_t bar;
  uint32_t phase;
  volatile int* abort_flag;
  unsigned* err;
  unsigned long long limit_ns;
};
__device__ __forceinline__ bool aux_wait(const AuxLoad& a) {
  if (mbar_try_wait(a.bar, a.phase)) return true;
  const unsigned long long t0 = global_ns();
  while (!mbar_try_wait(a.bar, a.phase)) {
    if (*a.abort_flag) return false;
    if (global_ns() - t0 > a.limit_ns) {
      *a.abort_flag = 1;
      atomicOr(a.err, kErrTimeout);
      return false;
    }
  }
  return true;
}
__device__ __forceinline__ void tma_store_2d(uint64_t map, uint32_t src, int c0, int c1) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(map),
               "r"(src), "r"(c0), "r"(c1)
               : "memory");
}
// Stores a 32 x 32 chunk (rows row0.., columns n..).  With a store map the
// chunk goes out as bulk tensor stores from the stage (its 64-byte rows in
// the 64-byte swizzle the map expects; rows and columns past the matrix are
// clipped by the copy); otherwise the lanes store the stage's rows.
__device__ __forceinline__ void stage_store_rows(uint4* st, void* base, int out_type, int64_t ld,
                                                 int row0, int M, int n, const float* v, int lane,
                                                 uint64_t map) {
  stage_acquire(lane);
  if (map != 0) {
    const uint32_t sbase = smem_addr(st);
    if (out_type == OUT_BF16) {
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint4 w;
        w.x = pack_bf16x2(v[8 * c + 0], v[8 * c + 1]);
        w.y = pack_bf16x2(v[8 * c + 2], v[8 * c + 3]);
        w.z = pack_bf16x2(v[8 * c + 4], v[8 * c + 5]);
        w.w = pack_bf16x2(v[8 * c + 6], v[8 * c + 7]);
        st[lane * 4 + (c ^ ((lane >> 1) & 3))] = w;
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) {
        tma_store_2d(map, sbase, n, row0);
        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
      }
    } else {
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        if (hh == 1) stage_acquire(lane);
#pragma unroll
        for (int c = 0; c < 4; ++c)
          st[lane * 4 + (c ^ ((lane >> 1) & 3))] =
              make_uint4(__float_as_uint(v[16 * hh + 4 * c + 0]), __float_as_uint(v[16 * hh + 4 * c + 1]),
                         __float_as_uint(v[16 * hh + 4 * c + 2]), __float_as_uint(v[16 * hh + 4 * c + 3]));
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(map, sbase, n + 16 * hh, row0);
          asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        }
      }
    }
    __syncwarp();
    return;
  }
  if (out_type == OUT_BF16) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint4 w;
      w.x = pack_bf16x2(v[8 * c + 0], v[8 * c + 1]);
      w.y = pack_bf16x2(v[8 * c + 2], v[8 * c + 3]);
      w.z = pack_bf16x2(v[8 * c + 4], v[8 * c + 5]);
      w.w = pack_bf16x2(v[8 * c + 6], v[8 * c + 7]);
      st[lane * 4 + (c ^ ((lane >> 1) & 3))] = w;
    }
    __syncwarp();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = i * 8 + (lane >> 2), c = lane & 3;
      const uint4 w = st[r * 4 + (c ^ ((r >> 1) & 3))];
      if (row0 + r < M)
        *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(base) +
                                  static_cast<int64_t>(row0 + r) * ld + n + c * 8) = w;
    }
  } else {
    // two 16-column halves, each 32 rows x 64 bytes
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
      for (int c = 0; c < 4; ++c)
        st[lane * 4 + (c ^ ((lane >> 1) & 3))] =
            make_uint4(__float_as_uint(v[16 * hh + 4 * c + 0]), __float_as_uint(v[16 * hh + 4 * c + 1]),
                       __float_as_uint(v[16 * hh + 4 * c + 2]), __float_as_uint(v[16 * hh + 4 * c + 3]));
      __syncwarp();
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int r = i * 8 + (lane >> 2), c = lane & 3;
        const uint4 w = st[r * 4 + (c ^ ((r >> 1) & 3))];
        if (row0 + r < M)
          *reinterpret_cast<uint4*>(static_cast<float*>(base) + static_cast<int64_t>(row0 + r) * ld +
                                    n + 16 * hh + c * 4) = w;
      }
      __syncwarp();
    }
  }
  __syncwarp();
}

// 32 x 32 bf16 chunk of the auxiliary operand through one bulk tensor load
// (rows past the matrix read as zeros); lane l then holds row row0 + l.
__device__ __forceinline__ void stage_load_aux_tma(uint4* st, uint64_t map, AuxLoad& a, int row0, int n,
                                                   float* z, int lane) {
  stage_acquire(lane);
  if (lane == 0) {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    mbar_arrive_expect_tx(a.bar, 32 * 64);
    tma_load_2d(smem_addr(st), map, a.bar, n, row0);
  }
  aux_wait(a);
  a.phase ^= 1u;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint4 w = st[lane * 4 + (c ^ ((lane >> 1) & 3))];
    unpack_bf16x2(w.x, z[8 * c + 0], z[8 * c + 1]);
    unpack_bf16x2(w.y, z[8 * c + 2], z[8 * c + 3]);
    unpack_bf16x2(w.z, z[8 * c + 4], z[8 * c + 5]);
    unpack_bf16x2(w.w, z[8 * c + 6], z[8 * c + 7]);
  }
  __syncwarp();
}
__device__ __forceinline__ void stage_load_rows_bf16(uint4* st, const void* base, int64_t ld,
                                                     int row0, int M, int n, float* z, int lane) {
  stage_acquire(lane);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = i * 8 + (lane >> 2), c = lane & 3;
    uint4 w = make_uint4(0, 0, 0, 0);
    if (row0 + r < M)
      w = __ldg(reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(base) +
                                               static_cast<int64_t>(row0 + r) * ld + n + c * 8));
    st[r * 4 + (c ^ ((r >> 1) & 3))] = w;
  }
  __syncwarp();
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint4 w = st[lane * 4 + (c ^ ((lane >> 1) & 3))];
    unpack_bf16x2(w.x, z[8 * c + 0], z[8 * c + 1]);
    unpack_bf16x2(w.y, z[8 * c + 2], z[8 * c + 3]);
    unpack_bf16x2(w.z, z[8 * c + 4], z[8 * c + 5]);
    unpack_bf16x2(w.w, z[8 * c + 6], z[8 * c + 7]);
  }
  __syncwarp();
}

__device__ __forceinline__ void stage_add_rows_f32(uint4* st, const void* base, int64_t ld, int row0,
                                                   int M, int n, float* v, int lane) {
  stage_acquire(lane);
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = i * 8 + (lane >> 2), c = lane & 3;
      uint4 w = make_uint4(0, 0, 0, 0);
      if (row0 + r < M)
        w = *reinterpret_cast<const uint4*>(static_cast<const float*>(base) +
                                            static_cast<int64_t>(row0 + r) * ld + n + 16 * hh + c * 4);
      st[r * 4 + (c ^ ((r >> 1) & 3))] = w;
    }
    __syncwarp();
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint4 w = st[lane * 4 + (c ^ ((lane >> 1) & 3))];
      v[16 * hh + 4 * c + 0] += __uint_as_float(w.x);
      v[16 * hh + 4 * c + 1] += __uint_as_float(w.y);
      v[16 * hh + 4 * c + 2] += __uint_as_float(w.z);
      v[16 * hh + 4 * c + 3] += __uint_as_float(w.w);
    }
    __syncwarp();
  }
}

// Pulls the bias of a warp's columns [n, n + 64) into L1 while the tile's
// main loop runs, so the epilogue's per-chunk bias reads do not wait on L2.
__device__ __forceinline__ void prefetch_bias(const GemmGroup& G, int n, int lane) {
  if (G.bias != nullptr && lane < 2 && n < G.N) {
    const int c = min(n + 63 * lane, G.N - 1);
    asm volatile("prefetch.global.L1 [%0];" ::"l"(static_cast<const __nv_bfloat16*>(G.bias) + c));
  }
}

// Epilogue of one 32 x 32 chunk: rows row0 .. row0+31 (lane l owns row0 + l),
// columns n .. n+31.  Called by all 32 lanes of the warp (the staged paths
// are warp-collective); rows >= M are computed but never stored.
template <bool ATTN>
__device__ __forceinline__ void epilogue_chunk(const GemmGroup& G, const CUtensorMap* mapO, uint4* st,
                                               AuxLoad& ax, int lane, int row0, int n, float* v) {
  // bulk-store maps of the group's outputs (0: the lanes store), bulk-load map of its operand
  const uint64_t map1 = G.out_map >= 0 ? reinterpret_cast<uint64_t>(mapO + G.out_map) : 0ull;
  const uint64_t map2 = G.out2_map >= 0 ? reinterpret_cast<uint64_t>(mapO + G.out2_map) : 0ull;
  const uint64_t mapx = G.aux_map >= 0 ? reinterpret_cast<uint64_t>(mapO + G.aux_map) : 0ull;
  const int row = row0 + lane;
  const bool row_ok = row < G.M;
  const int ncols = min(32, G.N - n);
  const bool coal = (ncols == 32) && G.vec_ok;  // warp-uniform
  if constexpr (ATTN) {
    if (G.epi == EPI_SMAX_BWD) {
      // dS = P * (dP - D) * alpha with P = aux, D = row_lse (the row's sum of P dP)
      float z[32];
      if (coal) {
        if (mapx != 0) stage_load_aux_tma(st, mapx, ax, row0, n, z, lane);
        else stage_load_rows_bf16(st, G.aux, G.ld_aux, row0, G.M, n, z, lane);
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) z[j] = 0.f;
        if (row_ok)
          load_bf16_chunk(static_cast<const __nv_bfloat16*>(G.aux) +
                              static_cast<int64_t>(row) * G.ld_aux + n,
                          z, ncols, false);
      }
      const float dd = row_ok ? G.row_lse[row] : 0.f;
      if (G.drop_mask != nullptr) {
        // attention dropout: dP = (dC V^T) * keep * scale
        const uint32_t keep = row_ok ? G.drop_mask[static_cast<int64_t>(row) * G.drop_wpr + (n >> 5)] : 0u;
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = (keep >> j) & 1u ? v[j] * G.drop_scale : 0.f;
      }
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = z[j] * (v[j] - dd) * G.alpha;
      if (coal) {
        stage_store_rows(st, G.out, OUT_BF16, G.ldo, row0, G.M, n, v, lane, map1);
      } else if (row_ok) {
        store_chunk(G.out, OUT_BF16, G.ldo, row, n, v, ncols, false);
      }
      return;
    }
  }
  switch (G.epi) {
    case EPI_STORE:
    case EPI_BIAS_GELU: {
      if (G.bias != nullptr) {
        // same address in every lane; the line was prefetched at tile start
        float b[32];
        load_bf16_chunk(static_cast<const __nv_bfloat16*>(G.bias) + n, b, ncols, coal);
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] += b[j];
      }
      if (coal) {
        stage_store_rows(st, G.out, G.out_type, G.ldo, row0, G.M, n, v, lane, map1);
      } else if (row_ok) {
        store_chunk(G.out, G.out_type, G.ldo, row, n, v, ncols, false);
      }
      if (G.epi == EPI_BIAS_GELU) {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = gelu_f(v[j]);
        if (coal) {
          stage_store_rows(st, G.out2, G.out_type, G.ldo, row0, G.M, n, v, lane, map2);
        } else if (row_ok) {
          store_chunk(G.out2, G.out_type, G.ldo, row, n, v, ncols, false);
        }
      }
      break;
    }
    case EPI_DGELU: {
      float z[32];
      if (coal) {
        if (mapx != 0) stage_load_aux_tma(st, mapx, ax, row0, n, z, lane);
        else stage_load_rows_bf16(st, G.aux, G.ld_aux, row0, G.M, n, z, lane);
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) z[j] = 0.f;
        if (row_ok)
          load_bf16_chunk(static_cast<const __nv_bfloat16*>(G.aux) +
                              static_cast<int64_t>(row) * G.ld_aux + n,
                          z, ncols, false);
      }
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] *= gelu_grad_f(z[j]);
      if (coal) {
        stage_store_rows(st, G.out, G.out_type, G.ldo, row0, G.M, n, v, lane, map1);
      } else if (row_ok) {
        store_chunk(G.out, G.out_type, G.ldo, row, n, v, ncols, false);
      }
      break;
    }
    case EPI_CE_BWD: {
      // dlogit = (softmax - onehot(target)) * dloss, softmax = 2^((acc - lse) log2 e)
      float lse = 0.f, dl = 0.f;
      int64_t tgt = -1;
      if (row_ok) {
        lse = G.row_lse[row];
        dl = G.row_dloss[row];
        tgt = G.row_target[row] - G.col0;
        tgt = tgt < G.N ? tgt - n : -1;  // a target in a later range is no column here
      }
      const float l2e = 1.4426950408889634f;
      const float base = -lse * l2e;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        float pj = ex2_ftz(fmaf(v[j], l2e, base));
        if (tgt == j) pj -= 1.f;
        v[j] = pj * dl;
      }
      if (coal) {
        stage_store_rows(st, G.out, OUT_BF16, G.ldo, row0, G.M, n, v, lane, map1);
      } else if (row_ok) {
        store_chunk(G.out, OUT_BF16, G.ldo, row, n, v, ncols, false);
      }
      break;
    }
    case EPI_F32:
    case EPI_SEGSUM: {
      if (G.epi == EPI_SEGSUM && row_ok) {
        const int64_t id = G.seg_row0 + row;
        const int b = G.seg_offsets[id], e = G.seg_offsets[id + 1];
        // the segment's rows added in position order, 16 columns at a time
        for (int t = b; t < e; ++t) {
          const __nv_bfloat16* src = static_cast<const __nv_bfloat16*>(G.seg_src) +
                                     static_cast<int64_t>(G.seg_perm[t]) * G.ld_seg + n;
          if (coal) {
            const uint4* s4 = reinterpret_cast<const uint4*>(src);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const uint4 w = __ldg(s4 + q);
              float x0, x1;
              unpack_bf16x2(w.x, x0, x1); v[8 * q + 0] += x0; v[8 * q + 1] += x1;
              unpack_bf16x2(w.y, x0, x1); v[8 * q + 2] += x0; v[8 * q + 3] += x1;
              unpack_bf16x2(w.z, x0, x1); v[8 * q + 4] += x0; v[8 * q + 5] += x1;
              unpack_bf16x2(w.w, x0, x1); v[8 * q + 6] += x0; v[8 * q + 7] += x1;
            }
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (j < ncols) v[j] += bf2f(src[j]);
          }
        }
      }
      if (coal) {
        if (G.accumulate) stage_add_rows_f32(st, G.out, G.ldo, row0, G.M, n, v, lane);
        stage_store_rows(st, G.out, OUT_F32, G.ldo, row0, G.M, n, v, lane, map1);
      } else if (row_ok) {
        float* o = static_cast<float*>(G.out) + static_cast<int64_t>(row) * G.ldo + n;
        if (G.accumulate) {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (j < ncols) v[j] += o[j];
        }
        store_chunk(G.out, OUT_F32, G.ldo, row, n, v, ncols, false);
      }
      break;
    }
    default:
      break;
  }
}

// ---------------------------------------------------------------------------
// Producer main loop of one segment, specialised on the operand forms:
// A_MODE 0 = K-major box, 1 = MN-major (two 64-wide boxes), 2 = MN-major 3D box;
// B_MODE 0 = K-major box, 1 = MN-major (N / 64 boxes), 2 = MN-major 3D box,
// 3 = the fixed ones block.  Keeping the form out of the loop leaves the loop
// body a straight line of TMA issues, which measured markedly faster than
// branching on the form every k-block.
// ---------------------------------------------------------------------------
struct ProdRing {
  uint32_t tiles_base, full0, empty0;  // smem addresses: stage 0 data, full[0], empty[0]
  int stage;
  uint32_t phase;
  uint32_t pend_valid, pend_phase;     // stages with a copy issued, and its phase
  bool skip_first;                     // fault injection: leave the first stage unfilled
};

template <int STAGES_, int STAGE_BYTES_, int A_MODE, int B_MODE>
__device__ __forceinline__ bool produce_kblocks(ProdRing& R, const WaitCtx& wctx, uint64_t mapA,
                                                uint64_t mapB, int kb0, int kb1, int m0, int n0,
                                                int n_mma) {
  const uint32_t stage_bytes = A_TILE_BYTES + static_cast<uint32_t>(n_mma) * BK * 2;
  for (int kb = kb0; kb < kb1; ++kb) {
    if (!wait_bounded(R.empty0 + 8u * R.stage, R.phase ^ 1u, wctx)) return false;
    const uint32_t a_dst = R.tiles_base + R.stage * STAGE_BYTES_;
    const uint32_t b_dst = a_dst + A_TILE_BYTES;
    const uint32_t fb = R.full0 + 8u * R.stage;
    if (R.skip_first) {
      R.skip_first = false;  // this stage is never filled; the consumer's wait expires
    } else {
      mbar_arrive_expect_tx(fb, stage_bytes);
      R.pend_valid |= 1u << R.stage;
      R.pend_phase = (R.pend_phase & ~(1u << R.stage)) | (R.phase << R.stage);
      const int k0 = kb * BK;
      if (A_MODE == 0) {
        tma_load_2d(a_dst, mapA, fb, k0, m0);
      } else if (A_MODE == 2) {
        tma_load_3d(a_dst, mapA, fb, 0, k0, m0 / 64);
      } else {
        tma_load_2d(a_dst, mapA, fb, m0, k0);
        tma_load_2d(a_dst + MN_BOX_BYTES, mapA, fb, m0 + 64, k0);
      }
      if (B_MODE == 0) {
        tma_load_2d(b_dst, mapB, fb, k0, n0);
      } else if (B_MODE == 2) {
        tma_load_3d(b_dst, mapB, fb, 0, k0, n0 / 64);
      } else if (B_MODE == 3) {
        tma_load_2d(b_dst, mapB, fb, 0, 0);
      } else {
        for (int j = 0; j < n_mma / 64; ++j)
          tma_load_2d(b_dst + j * MN_BOX_BYTES, mapB, fb, n0 + 64 * j, k0);
      }
    }
    if (++R.stage == STAGES_) {
      R.stage = 0;
      R.phase ^= 1u;
    }
  }
  return true;
}

template <int STAGES_, int STAGE_BYTES_>
__device__ __forceinline__ bool produce_segment(ProdRing& R, const WaitCtx& wctx, const TcSeg& S,
                                                uint64_t mapA, uint64_t mapB, int kb0, int kb1,
                                                int m0, int n0) {
  const int a_mode = S.a_3d ? 2 : (S.a_mn ? 1 : 0);
  const int b_mode = S.b_fixed ? 3 : (S.b_3d ? 2 : (S.b_mn ? 1 : 0));
  const int n_mma = S.n_mma;
#define TP_PRODUCE(am, bm) \
  produce_kblocks<STAGES_, STAGE_BYTES_, am, bm>(R, wctx, mapA, mapB, kb0, kb1, m0, n0, n_mma)
  switch (a_mode * 4 + b_mode) {
    case 0: return TP_PRODUCE(0, 0);
    case 1: return TP_PRODUCE(0, 1);
    case 2: return TP_PRODUCE(0, 2);
    case 3: return TP_PRODUCE(0, 3);
    case 4: return TP_PRODUCE(1, 0);
    case 5: return TP_PRODUCE(1, 1);
    case 6: return TP_PRODUCE(1, 2);
    case 7: return TP_PRODUCE(1, 3);
    case 8: return TP_PRODUCE(2, 0);
    case 9: return TP_PRODUCE(2, 1);
    case 10: return TP_PRODUCE(2, 2);
    default: return TP_PRODUCE(2, 3);
  }
#undef TP_PRODUCE
}

// ---------------------------------------------------------------------------
// Cross-entropy forward epilogue of one warp's region: its 32 rows (lane =
// row) and 64 columns [n0 + 32 c_begin, +64), one "part" of the row.  The
// logits stay in TMEM and registers: the warp writes the part's (max, sum of
// exp(logit - max)) per row, and the logit at the row's target column when
// the target lies in the part.
// ---------------------------------------------------------------------------
template <bool ATTN>
__device__ __forceinline__ void ce_fwd_epilogue_warp(const GemmGroup& G, int lane, int row0, int n0,
                                                     int c_begin, int cpw, uint32_t taddr) {
  const int nb = n0 + c_begin * 32;
  if (nb >= G.N) return;  // warp-uniform: no part here
  const int row = row0 + lane;
  const bool row_ok = row < G.M;
  int64_t tgt = (row_ok && G.row_target) ? G.row_target[row] - G.col0 : -1;
  if (tgt >= G.N) tgt = -1;  // the target is in a later range (the tile's zero-filled columns)
  const float l2e = 1.4426950408889634f;
  const float alpha = ATTN ? G.alpha : 1.f;
  float m = -INFINITY, s = 0.f;
  for (int c = c_begin; c < c_begin + cpw; ++c) {
    const int n = n0 + c * 32;
    if (n >= G.N) break;  // warp-uniform
    // columns j < jn of this chunk count (causal: key n + j <= query row)
    const int jn = (ATTN && G.causal) ? min(min(32, G.N - n), row - n + 1) : min(32, G.N - n);
    uint32_t rr[32];
    tmem_ld32(taddr + static_cast<uint32_t>(c * 32), rr);
    float x[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) x[j] = ATTN ? __uint_as_float(rr[j]) * alpha : __uint_as_float(rr[j]);
    float mx = -INFINITY;
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (j < jn) mx = fmaxf(mx, x[j]);
    const int64_t tj = tgt - n;
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (tj == j && row_ok) G.ce_target[row] = x[j];
    const float nm = fmaxf(m, mx);
    if (ATTN && nm == -INFINITY) continue;  // nothing counted yet in this row
    float acc = s * ex2_ftz((m - nm) * l2e);
    const float base = -nm * l2e;
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (j < jn) acc += ex2_ftz(fmaf(x[j], l2e, base));
    m = nm;
    s = acc;
  }
  if (row_ok) {
    const int64_t part = G.ce_part0 + nb / 64;
    reinterpret_cast<float2*>(G.ce_part)[part * G.ce_rows + row] = make_float2(m, s);
  }
}

// ---------------------------------------------------------------------------
// Attention scores epilogue of one warp's region (its 32 rows and one 64-column
// part, as above): m = the part's max of alpha acc over the columns the causal
// mask keeps, e = exp(alpha acc - m) stored in bf16 (0 where masked), and
// (m, sum e) per row to the part statistics.  A first pass over the part's
// TMEM columns finds m, a second computes, sums and stores e.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void smax_parts_epilogue_warp(const GemmGroup& G, const CUtensorMap* mapO,
                                                         uint4* st, int lane, int row0, int n0, int c_begin,
                                                         int cpw, uint32_t taddr) {
  const int nb = n0 + c_begin * 32;
  if (nb >= G.N) return;  // warp-uniform: no part here
  const int row = row0 + lane;
  const bool row_ok = row < G.M;
  const uint64_t map1 = G.out_map >= 0 ? reinterpret_cast<uint64_t>(mapO + G.out_map) : 0ull;
  const float l2e = 1.4426950408889634f;
  float m = -INFINITY;
  for (int c = c_begin; c < c_begin + cpw; ++c) {
    const int n = n0 + c * 32;
    if (n >= G.N) break;  // warp-uniform
    const int jn = G.causal ? min(min(32, G.N - n), row - n + 1) : min(32, G.N - n);
    uint32_t rr[32];
    tmem_ld32(taddr + static_cast<uint32_t>(c * 32), rr);
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (j < jn) m = fmaxf(m, __uint_as_float(rr[j]) * G.alpha);
  }
  const float base = m == -INFINITY ? 0.f : -m * l2e;  // a row with no kept column stores zeros
  float sum = 0.f;
  for (int c = c_begin; c < c_begin + cpw; ++c) {
    const int n = n0 + c * 32;
    if (n >= G.N) break;  // warp-uniform
    const int ncols = min(32, G.N - n);
    const int jn = G.causal ? min(ncols, row - n + 1) : ncols;
    uint32_t rr[32];
    tmem_ld32(taddr + static_cast<uint32_t>(c * 32), rr);
    float v[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      v[j] = j < jn ? ex2_ftz(fmaf(__uint_as_float(rr[j]) * G.alpha, l2e, base)) : 0.f;
      sum += v[j];
    }
    if (ncols == 32 && G.vec_ok) {
      stage_store_rows(st, G.out, OUT_BF16, G.ldo, row0, G.M, n, v, lane, map1);
    } else if (row_ok) {
      store_chunk(G.out, OUT_BF16, G.ldo, row, n, v, ncols, false);
    }
  }
  if (row_ok) {
    const int64_t part = G.ce_part0 + nb / 64;
    reinterpret_cast<float2*>(G.ce_part)[part * G.ce_rows + row] = make_float2(m, sum);
  }
}

// ---------------------------------------------------------------------------
// Dynamic tile scheduling: one (next, done) counter pair per launch slot.  The
// last CTA to finish resets its pair, so the next launch using the slot starts
// from zero.  Launches rotate over the slots.
// ---------------------------------------------------------------------------
constexpr int kSchedSlots = 64;
__device__ int g_sched[2 * kSchedSlots];
__device__ int g_dep[kSchedSlots * kMaxCounters];

// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------
template <bool ATTN>
__global__ void __launch_bounds__(NUM_THREADS, 1) tc_gemm_kernel(const __grid_constant__ TcGemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  // bars: full[S], empty[S], tfull[2], tempty[2], drain, tile_full[R], tile_empty[R]
  constexpr int kBarCount = 2 * STAGES + 5 + 2 * TILE_RING;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kBarCount);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + kBarCount + 1);
  // tile ring: (tile id or -1, group, m0, n0) per slot, decoded once by the producer
  volatile int* tile_ids = reinterpret_cast<volatile int*>(bars + kBarCount + 2);
  // one mbarrier per epilogue warp for its auxiliary-operand loads
  uint64_t* aux_bars = bars + kBarCount + 2 + 2 * TILE_RING;
  static_assert((kBarCount + 2 + 2 * TILE_RING + NUM_EPI_WARPS) * 8 <= BAR_BYTES, "barrier area");
  GrpLite* gtab = reinterpret_cast<GrpLite*>(smem + STAGES * STAGE_BYTES + BAR_BYTES +
                                             NUM_EPI_WARPS * EPI_WARP_BYTES);
  fill_group_table(p, gtab, threadIdx.x, NUM_THREADS);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t bar0 = smem_addr(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + b); };
  auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + 2 + b); };
  const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 4);
  auto tile_full_bar = [&](int r) { return bar0 + 8u * (2 * STAGES + 5 + r); };
  auto tile_empty_bar = [&](int r) { return bar0 + 8u * (2 * STAGES + 5 + TILE_RING + r); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), NUM_EPI_WARPS);
    }
    mbar_init(drain_bar, 1);
    for (int r = 0; r < TILE_RING; ++r) {
      mbar_init(tile_full_bar(r), 1);
      mbar_init(tile_empty_bar(r), 1 + NUM_EPI_WARPS);
    }
    for (int w = 0; w < NUM_EPI_WARPS; ++w) mbar_init(smem_addr(aux_bars + w), 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(tmem_slot)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // set-up done: wait until the previous kernel on the stream has completed
  pdl_wait();

  const WaitCtx wctx{abort_flag, p.err, p.wait_limit_ns};
  const uint32_t tiles_base = smem_addr(smem);
  int* sched = g_sched + 2 * p.sched_slot;
  int* dep = g_dep + kMaxCounters * p.sched_slot;

  if (warp == 0 && lane == 0) {
    // ---------------------- tile scheduler + TMA producer ----------------------
    for (int s = 0; s < p.num_segs; ++s) {
      prefetch_tmap(&p.mapA[s]);
      prefetch_tmap(&p.mapB[s]);
    }
    ProdRing R{tiles_base, full_bar(0), empty_bar(0), 0, 0u, 0u, 0u, p.fault_skip != 0};
    // Hot-loop values live in registers: reading the kernel parameters
    // through references re-loads them after every asm statement.
    const int total_tiles = p.total_tiles;
    const bool claim_ahead = !p.has_dep;
    bool ok = true;
    int tile = blockIdx.x;
    for (int i = 0; ok; ++i) {
      // publish the tile id (or -1 = done) to the other roles
      const int r = i % TILE_RING;
      if (!wait_bounded(tile_empty_bar(r), static_cast<uint32_t>((i / TILE_RING) & 1) ^ 1u, wctx)) break;
      const int t = tile < total_tiles ? tile : -1;
      TileCoord tc{0, 0, 0};
      if (t >= 0) tc = decode_tile_rows<BM, ATTN>(p, gtab, t);
      tile_ids[4 * r] = t;
      tile_ids[4 * r + 1] = tc.g;
      tile_ids[4 * r + 2] = tc.m0;
      tile_ids[4 * r + 3] = tc.n0;
      mbar_arrive(tile_full_bar(r));
      if (t < 0) {
        pdl_trigger();  // no tile left for this CTA: the next kernel may launch
        break;
      }
      // Next tile: the first gridDim tiles are static, the rest claimed in
      // order.  Without dependent tiles the claim is made now, so its atomic
      // round trip overlaps this tile's loads; with them it waits until this
      // tile's loads are issued (a held tile would sit behind a dependency wait).
      int next = -1;
      if (claim_ahead) next = static_cast<int>(gridDim.x) + atomicAdd(sched, 1);
      const GemmGroup& G = p.grp[tc.g];
      const int seg_begin = G.seg_begin, seg_end = G.seg_end;
      if (G.dep_kind != DEP_NONE) {
        // wait (bounded) until the tiles this one reads have been stored
        const int* ctr = dep + G.dep_base + (G.dep_kind == DEP_ROW ? tc.m0 / BM : tc.m0 / BN);
        if (ld_acquire_gpu(ctr) < G.dep_target) {
          const unsigned long long t0 = global_ns();
          while (ld_acquire_gpu(ctr) < G.dep_target) {
            if (*abort_flag) {
              ok = false;
              break;
            }
            if (global_ns() - t0 > p.wait_limit_ns) {
              *abort_flag = 1;
              atomicOr(p.err, kErrTimeout);
              ok = false;
              break;
            }
            __nanosleep(128);
          }
        }
        // order the TMA (async proxy) reads after the acquire
        asm volatile("fence.proxy.async.global;" ::: "memory");
      }
      for (int s = seg_begin; ok && s < seg_end; ++s) {
        const TcSeg S = p.seg[s];
        int kb0, kb1;
        tile_kb_range<BM, ATTN>(G, S.K, tc.m0, tc.n0, kb0, kb1);
        ok = produce_segment<STAGES, STAGE_BYTES>(R, wctx, S, reinterpret_cast<uint64_t>(&p.mapA[s]),
                                                  reinterpret_cast<uint64_t>(&p.mapB[s]), kb0, kb1,
                                                  tc.m0, tc.n0);
      }
      // next tile: the first gridDim tiles are static, the rest claimed in order
      tile = claim_ahead ? next : static_cast<int>(gridDim.x) + atomicAdd(sched, 1);
    }
    if (*abort_flag) {
      // Drain: wait (bounded) until every copy this thread issued has landed.
      for (int s = 0; s < STAGES; ++s) {
        if (!((R.pend_valid >> s) & 1u)) continue;
        const unsigned long long t0 = global_ns();
        while (!mbar_try_wait(full_bar(s), (R.pend_phase >> s) & 1u)) {
          if (global_ns() - t0 > p.wait_limit_ns) break;
        }
      }
    }
  } else if (warp == 1 && lane == 0) {
    // ------------------------------- MMA issuer -------------------------------
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    bool issued_any = false;
    for (int lt = 0; ok; ++lt) {
      const int r = lt % TILE_RING;
      if (!wait_bounded(tile_full_bar(r), static_cast<uint32_t>((lt / TILE_RING) & 1), wctx)) break;
      const int tile = tile_ids[4 * r];
      const TileCoord tc{tile_ids[4 * r + 1], tile_ids[4 * r + 2], tile_ids[4 * r + 3]};
      mbar_arrive(tile_empty_bar(r));
      if (tile < 0) break;
      const GemmGroup& G = p.grp[tc.g];
      const int buf = lt & 1;
      const uint32_t tphase = static_cast<uint32_t>(lt >> 1) & 1u;
      if (!wait_bounded(tempty_bar(buf), tphase ^ 1u, wctx)) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * BN);
      const int seg_begin = G.seg_begin, seg_end = G.seg_end;
      uint32_t acc = 0;
      for (int s = seg_begin; ok && s < seg_end; ++s) {
        const TcSeg S = p.seg[s];
        int kb0, kb1;
        tile_kb_range<BM, ATTN>(G, S.K, tc.m0, tc.n0, kb0, kb1);
        const uint32_t idesc = idesc_bf16(S.a_mn, S.b_mn, S.n_mma);
        // Descriptors of stage 0; a stage / k-step offset is added to the
        // 14-bit start-address field (shared addresses stay below 256 KB).
        // K-major: 16 K elements = 32 bytes along the swizzled row.
        // MN-major: 16 K rows = 2 swizzle atoms of 8 rows x 128 bytes.
        const uint64_t a_desc0 = sdesc(tiles_base, S.a_mn ? MN_BOX_BYTES : 16, 1024);
        const uint64_t b_desc0 = sdesc(tiles_base + A_TILE_BYTES, S.b_mn ? MN_BOX_BYTES : 16, 1024);
        const uint32_t a_step = S.a_mn ? (2048 >> 4) : (32 >> 4);
        const uint32_t b_step = S.b_mn ? (2048 >> 4) : (32 >> 4);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!wait_bounded(full_bar(stage), phase, wctx)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t off = static_cast<uint32_t>(stage * STAGE_BYTES) >> 4;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            mma_bf16(d_tmem, a_desc0 + off + kk * a_step, b_desc0 + off + kk * b_step, idesc, acc);
            acc = 1;
          }
          issued_any = true;
          mma_commit(empty_bar(stage));
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) break;
      mma_commit(tfull_bar(buf));
    }
    if (*abort_flag && issued_any) {
      // Drain: the commit arrives once every MMA issued so far has completed.
      mma_commit(drain_bar);
      const unsigned long long t0 = global_ns();
      while (!mbar_try_wait(drain_bar, 0)) {
        if (global_ns() - t0 > p.wait_limit_ns) break;
      }
    }
  } else if (warp >= 2) {
    // -------------------------------- Epilogue --------------------------------
    const int quarter = warp & 3;              // TMEM lanes this warp may access
    uint4* epi_stage = reinterpret_cast<uint4*>(smem + STAGES * STAGE_BYTES + BAR_BYTES +
                                                (warp - 2) * EPI_WARP_BYTES);
    const int part = (warp - 2) >> 2;  // which quarter of the tile's columns
    AuxLoad ax{smem_addr(aux_bars + (warp - 2)), 0u, abort_flag, p.err, p.wait_limit_ns};
    for (int lt = 0;; ++lt) {
      const int r = lt % TILE_RING;
      if (!wait_bounded(tile_full_bar(r), static_cast<uint32_t>((lt / TILE_RING) & 1), wctx)) break;
      const int tile = tile_ids[4 * r];
      const TileCoord tc{tile_ids[4 * r + 1], tile_ids[4 * r + 2], tile_ids[4 * r + 3]};
      __syncwarp();
      if (lane == 0) mbar_arrive(tile_empty_bar(r));
      if (tile < 0) break;
      const GemmGroup& G = p.grp[tc.g];
      const int buf = lt & 1;
      const uint32_t tphase = static_cast<uint32_t>(lt >> 1) & 1u;
      const int cpw = G.bn / (32 * EPI_PARTS);  // 32-column chunks per warp
      const int c_begin = part * cpw;
      prefetch_bias(G, tc.n0 + c_begin * 32, lane);
      if (!wait_bounded(tfull_bar(buf), tphase, wctx)) break;
      tc_fence_after();
      const int row0 = tc.m0 + quarter * 32;
      const uint32_t taddr =
          tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(buf * BN);
      const bool empty = tile_empty<BM, ATTN>(p, G, tc.m0, tc.n0);
      if (G.epi == EPI_CE_FWD) ce_fwd_epilogue_warp<ATTN>(G, lane, row0, tc.n0, c_begin, cpw, taddr);
      if (ATTN && G.epi == EPI_SMAX_PARTS)
        smax_parts_epilogue_warp(G, p.mapO, epi_stage, lane, row0, tc.n0, c_begin, cpw, taddr);
      for (int c = c_begin; G.epi != EPI_CE_FWD && !(ATTN && G.epi == EPI_SMAX_PARTS) && c < c_begin + cpw;
           ++c) {
        const int n = tc.n0 + c * 32;
        if (n >= G.N) break;  // warp-uniform
        uint32_t rr[32];
        float v[32];
        if (empty) {
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = 0.f;
        } else {
          tmem_ld32(taddr + static_cast<uint32_t>(c * 32), rr);
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(rr[j]);
        }
        epilogue_chunk<ATTN>(G, p.mapO, epi_stage, ax, lane, row0, n, v);
      }
      tc_fence_before();
      if (G.prod_row >= 0 || G.prod_col >= 0) {
        // dependants read this tile: its bulk stores complete before the warp arrives
        if (lane == 0) {
          asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
          asm volatile("fence.proxy.async.global;" ::: "memory");
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty_bar(buf));
      if ((G.prod_row >= 0 || G.prod_col >= 0) && warp == 2 + lt % NUM_EPI_WARPS) {
        // One warp per tile (rotating) counts the tile for its dependants:
        // once every epilogue warp has arrived on tempty (release.cta after
        // its stores; this wait acquires), a GPU-scope fence and the counter
        // add publish all of the tile's stores.  The other warps move on
        // without a fence.
        if (lane == 0) {
          if (wait_bounded(tempty_bar(buf), tphase, wctx)) {
            __threadfence();
            if (G.prod_row >= 0) atomicAdd(dep + G.prod_row + tc.m0 / BM, 1);
            if (G.prod_col >= 0) atomicAdd(dep + G.prod_col + tc.n0 / BN, 1);
          }
        }
        __syncwarp();
      }
    }
  }

  // every bulk tensor store of the epilogue has finished before the CTA exits
  if (warp >= 2 && lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(TMEM_COLS)
                 : "memory");
  }
  if (threadIdx.x == 0) {
    // The last CTA to finish resets this launch slot's counters.
    __threadfence();
    if (atomicAdd(sched + 1, 1) == static_cast<int>(gridDim.x) - 1) {
      for (int c = 0; c < p.num_counters; ++c) atomicExch(dep + c, 0);
      atomicExch(sched, 0);
      atomicExch(sched + 1, 0);
    }
  }
}

// ===========================================================================
// Two-SM variant: a cluster of two CTAs computes a 256 x 256 tile with
// tcgen05.mma.cta_group::2.  Each CTA stages its own 128 rows of A and its own
// 128 columns of B, so a stage is 32 KB instead of 48 KB and six stages fit;
// the two SMs' tensor cores share one instruction issued by the leader
// (cluster rank 0).  Each CTA's TMEM holds the accumulator of its 128 rows,
// and each CTA runs the same epilogue as the one-SM kernel on its rows.
//
// Coordination (all waits bounded):
//   leader producer   claims tiles, writes each tile id into both CTAs' rings,
//                     expects both halves' bytes on its full[s]
//   both producers    TMA their halves into their own smem; the copies of
//                     both CTAs complete on the leader's full[s]
//   leader MMA        waits full[s], issues the pair MMA, commits (multicast
//                     to both CTAs) to empty[s] and to tfull[b]
//   both epilogues    read their TMEM rows, then arrive on the leader's tempty[b]
// A cluster barrier at the end keeps both CTAs' shared memory alive until
// neither touches the other's any more.
// ===========================================================================
constexpr int BM2 = 256;                           // rows per pair tile
constexpr int STAGES2 = 6;
constexpr int B_HALF_BYTES = 128 * BK * 2;          // 16 KB
constexpr int STAGE2_BYTES = A_TILE_BYTES + B_HALF_BYTES;
constexpr int SMEM2_BYTES =
    STAGES2 * STAGE2_BYTES + BAR_BYTES + NUM_EPI_WARPS * EPI_WARP_BYTES + TBL_BYTES + 1024;
static_assert(SMEM_BYTES <= 227 * 1024 && SMEM2_BYTES <= 227 * 1024,
              "dynamic shared memory above the 227 KB a CTA may use");

// TMA load into this CTA's shared memory whose completion is signalled on an
// mbarrier that may live in the peer CTA of the pair (cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, uint64_t map,
                                                 uint32_t bar_cluster, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(map), "r"(bar_cluster), "r"(c0), "r"(c1));
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Shared-memory address of the same object in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}

__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ void st_cluster_u32(uint32_t cluster_addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

struct WaitCtx2 {
  volatile int* abort_flag;
  uint32_t peer_abort;  // cluster address of the peer's abort flag
  unsigned* err;
  unsigned long long limit_ns;
};

__device__ __forceinline__ void raise_abort2(const WaitCtx2& w, bool timed_out) {
  *w.abort_flag = 1;
  st_cluster_u32(w.peer_abort, 1u);
  if (timed_out) atomicOr(w.err, kErrTimeout);
}

// Bounded wait with cluster-scope acquire (the phase may be completed by the
// peer CTA).  Returns false on abort or timeout.
__device__ __forceinline__ bool wait2(uint32_t bar, uint32_t parity, const WaitCtx2& w) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  while (true) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if (*w.abort_flag) return false;
    if (global_ns() - t0 > w.limit_ns) {
      raise_abort2(w, true);
      return false;
    }
  }
}

__device__ __forceinline__ void mma_bf16_pair(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                              uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
}

// Arrives on the mbarrier at `bar` in both CTAs of the pair once all prior
// MMAs of this thread have completed.
__device__ __forceinline__ void mma_commit_pair(uint32_t bar, uint16_t mask = 0x3) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"(mask)
      : "memory");
}

__device__ __forceinline__ uint32_t idesc_bf16_m256(int a_mn, int b_mn, int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(a_mn) << 15) |
         (static_cast<uint32_t>(b_mn) << 16) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(BM2 >> 4) << 24);
}

// Producer main loop of one segment for the two-SM kernel (same operand
// forms as produce_kblocks; each CTA loads its 128 rows of A and its half of
// B, and both CTAs' copies complete on the leader's full barrier).
template <int A_MODE, int B_MODE>
__device__ __forceinline__ bool produce_kblocks_pair(ProdRing& R, const WaitCtx2& wctx, bool leader,
                                                     uint64_t mapA, uint64_t mapB, int kb0, int kb1,
                                                     int row0, int ncol0, uint32_t b_bytes) {
  for (int kb = kb0; kb < kb1; ++kb) {
    if (!wait2(R.empty0 + 8u * R.stage, R.phase ^ 1u, wctx)) return false;
    const uint32_t a_dst = R.tiles_base + R.stage * STAGE2_BYTES;
    const uint32_t b_dst = a_dst + A_TILE_BYTES;
    if (R.skip_first) {
      R.skip_first = false;  // this stage is never filled; the consumer's wait expires
    } else {
      const uint32_t own_full = R.full0 + 8u * R.stage;
      const uint32_t fb = map_to_rank(own_full, 0);
      if (leader) {
        mbar_arrive_expect_tx(own_full, 2 * (A_TILE_BYTES + b_bytes));
        R.pend_valid |= 1u << R.stage;
        R.pend_phase = (R.pend_phase & ~(1u << R.stage)) | (R.phase << R.stage);
      }
      const int k0 = kb * BK;
      if (A_MODE == 0) {
        tma_load_2d_pair(a_dst, mapA, fb, k0, row0);
      } else if (A_MODE == 2) {
        tma_load_3d_pair(a_dst, mapA, fb, 0, k0, row0 / 64);
      } else {
        tma_load_2d_pair(a_dst, mapA, fb, row0, k0);
        tma_load_2d_pair(a_dst + MN_BOX_BYTES, mapA, fb, row0 + 64, k0);
      }
      if (B_MODE == 0) {
        tma_load_2d_pair(b_dst, mapB, fb, k0, ncol0);
      } else if (B_MODE == 2) {
        tma_load_3d_pair(b_dst, mapB, fb, 0, k0, ncol0 / 64);
      } else if (B_MODE == 3) {
        tma_load_2d_pair(b_dst, mapB, fb, 0, 0);
      } else {
        tma_load_2d_pair(b_dst, mapB, fb, ncol0, k0);
        tma_load_2d_pair(b_dst + MN_BOX_BYTES, mapB, fb, ncol0 + 64, k0);
      }
    }
    if (++R.stage == STAGES2) {
      R.stage = 0;
      R.phase ^= 1u;
    }
  }
  return true;
}

__device__ __forceinline__ bool produce_segment_pair(ProdRing& R, const WaitCtx2& wctx, bool leader,
                                                     const TcSeg& S, uint64_t mapA, uint64_t mapB,
                                                     int kb0, int kb1, int row0, int ncol0) {
  const int a_mode = S.a_3d ? 2 : (S.a_mn ? 1 : 0);
  const int b_mode = S.b_fixed ? 3 : (S.b_3d ? 2 : (S.b_mn ? 1 : 0));
  const uint32_t b_bytes = S.b_fixed ? static_cast<uint32_t>(S.n_mma / 2) * BK * 2 : B_HALF_BYTES;
#define TP_PRODUCE2(am, bm) \
  produce_kblocks_pair<am, bm>(R, wctx, leader, mapA, mapB, kb0, kb1, row0, ncol0, b_bytes)
  switch (a_mode * 4 + b_mode) {
    case 0: return TP_PRODUCE2(0, 0);
    case 1: return TP_PRODUCE2(0, 1);
    case 2: return TP_PRODUCE2(0, 2);
    case 3: return TP_PRODUCE2(0, 3);
    case 4: return TP_PRODUCE2(1, 0);
    case 5: return TP_PRODUCE2(1, 1);
    case 6: return TP_PRODUCE2(1, 2);
    case 7: return TP_PRODUCE2(1, 3);
    case 8: return TP_PRODUCE2(2, 0);
    case 9: return TP_PRODUCE2(2, 1);
    case 10: return TP_PRODUCE2(2, 2);
    default: return TP_PRODUCE2(2, 3);
  }
#undef TP_PRODUCE2
}

template <bool ATTN>
__global__ void __launch_bounds__(NUM_THREADS, 1) tc_gemm_pair_kernel(const __grid_constant__ TcGemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES2 * STAGE2_BYTES);
  // bars: full[S], empty[S], tfull[2], tempty[2], drain, tile_full[R], tile_empty[R]
  constexpr int kBarCount = 2 * STAGES2 + 5 + 2 * TILE_RING;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kBarCount);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + kBarCount + 1);
  // tile ring: (tile id or -1, group, m0, n0) per slot, decoded once by the leader's producer
  volatile int* tile_ids = reinterpret_cast<volatile int*>(bars + kBarCount + 2);
  // one mbarrier per epilogue warp for its auxiliary-operand loads
  uint64_t* aux_bars = bars + kBarCount + 2 + 2 * TILE_RING;
  static_assert((kBarCount + 2 + 2 * TILE_RING + NUM_EPI_WARPS) * 8 <= BAR_BYTES, "barrier area");
  GrpLite* gtab = reinterpret_cast<GrpLite*>(smem + STAGES2 * STAGE2_BYTES + BAR_BYTES +
                                             NUM_EPI_WARPS * EPI_WARP_BYTES);
  fill_group_table(p, gtab, threadIdx.x, NUM_THREADS);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const uint32_t peer = rank ^ 1u;
  const bool leader = rank == 0;
  const uint32_t bar0 = smem_addr(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES2 + s); };
  auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * STAGES2 + b); };
  auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * STAGES2 + 2 + b); };
  const uint32_t drain_bar = bar0 + 8u * (2 * STAGES2 + 4);
  auto tile_full_bar = [&](int r) { return bar0 + 8u * (2 * STAGES2 + 5 + r); };
  auto tile_empty_bar = [&](int r) { return bar0 + 8u * (2 * STAGES2 + 5 + TILE_RING + r); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES2; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), 2 * NUM_EPI_WARPS);
    }
    mbar_init(drain_bar, 1);
    for (int r = 0; r < TILE_RING; ++r) {
      mbar_init(tile_full_bar(r), 1);
      // leader: its MMA thread and epilogue warps; peer: its producer and epilogue warps
      mbar_init(tile_empty_bar(r), 2 * (1 + NUM_EPI_WARPS));
    }
    for (int w = 0; w < NUM_EPI_WARPS; ++w) mbar_init(smem_addr(aux_bars + w), 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(tmem_slot)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // both CTAs' barriers are initialised before any remote arrive
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // set-up done: wait until the previous kernel on the stream has completed
  pdl_wait();

  const WaitCtx2 wctx{abort_flag, map_to_rank(smem_addr(const_cast<int*>(abort_flag)), peer), p.err,
                      p.wait_limit_ns};
  const uint32_t tiles_base = smem_addr(smem);
  int* sched = g_sched + 2 * p.sched_slot;
  int* dep = g_dep + kMaxCounters * p.sched_slot;
  const uint32_t tile_ids_addr = smem_addr(const_cast<int*>(tile_ids));

  // Every role reads the i-th tile id from its CTA's ring, then releases the
  // slot on the leader's tile_empty barrier.
  auto take_tile = [&](int i, int& t, TileCoord& tc) -> bool {
    const int r = i % TILE_RING;
    if (!wait2(tile_full_bar(r), static_cast<uint32_t>((i / TILE_RING) & 1), wctx)) return false;
    t = tile_ids[4 * r];
    tc = TileCoord{tile_ids[4 * r + 1], tile_ids[4 * r + 2], tile_ids[4 * r + 3]};
    return true;
  };
  auto release_tile = [&](int i) {
    const int r = i % TILE_RING;
    if (leader) mbar_arrive(tile_empty_bar(r));
    else mbar_arrive_remote(map_to_rank(tile_empty_bar(r), 0));
  };

  if (warp == 0 && lane == 0) {
    // --------------- tile scheduler (leader) + TMA producer (both) ---------------
    for (int s = 0; s < p.num_segs; ++s) {
      prefetch_tmap(&p.mapA[s]);
      prefetch_tmap(&p.mapB[s]);
    }
    ProdRing R{tiles_base, full_bar(0), empty_bar(0), 0, 0u, 0u, 0u, p.fault_skip != 0};
    const int total_tiles = p.total_tiles;
    bool ok = true;
    int claim = blockIdx.x >> 1;  // the cluster's first tile
    const bool claim_ahead = !p.has_dep;
    for (int i = 0; ok; ++i) {
      int t;
      TileCoord tc{0, 0, 0};
      if (leader) {
        const int r = i % TILE_RING;
        if (!wait2(tile_empty_bar(r), static_cast<uint32_t>((i / TILE_RING) & 1) ^ 1u, wctx)) break;
        t = claim < total_tiles ? claim : -1;
        if (t >= 0) tc = decode_tile_rows<BM2, ATTN>(p, gtab, t);
        const int vals[4] = {t, tc.g, tc.m0, tc.n0};
        for (int q = 0; q < 4; ++q) {
          tile_ids[4 * r + q] = vals[q];
          st_cluster_u32(map_to_rank(tile_ids_addr + 4u * (4 * r + q), peer), static_cast<uint32_t>(vals[q]));
        }
        mbar_arrive(tile_full_bar(r));
        mbar_arrive_remote(map_to_rank(tile_full_bar(r), peer));
      } else {
        if (!take_tile(i, t, tc)) break;
        release_tile(i);
      }
      if (t < 0) {
        pdl_trigger();  // no tile left for this CTA: the next kernel may launch
        break;
      }
      // the leader claims the cluster's next tile (ahead when nothing waits; see the one-SM kernel)
      int next = -1;
      if (leader && claim_ahead) next = static_cast<int>(gridDim.x >> 1) + atomicAdd(sched, 1);
      const GemmGroup& G = p.grp[tc.g];
      const int seg_begin = G.seg_begin, seg_end = G.seg_end;
      const int row0 = tc.m0 + 128 * static_cast<int>(rank);  // this CTA's rows
      if (G.dep_kind != DEP_NONE) {
        const int* ctr = dep + G.dep_base + (G.dep_kind == DEP_ROW ? row0 / BM : tc.m0 / BN);
        if (ld_acquire_gpu(ctr) < G.dep_target) {
          const unsigned long long t0 = global_ns();
          while (ld_acquire_gpu(ctr) < G.dep_target) {
            if (*abort_flag) {
              ok = false;
              break;
            }
            if (global_ns() - t0 > p.wait_limit_ns) {
              raise_abort2(wctx, true);
              ok = false;
              break;
            }
            __nanosleep(128);
          }
        }
        asm volatile("fence.proxy.async.global;" ::: "memory");
      }
      const int ncol0 = tc.n0 + 128 * static_cast<int>(rank);  // this CTA's half of B
      for (int s = seg_begin; ok && s < seg_end; ++s) {
        const TcSeg S = p.seg[s];
        int kb0, kb1;
        tile_kb_range<BM2, ATTN>(G, S.K, tc.m0, tc.n0, kb0, kb1);
        ok = produce_segment_pair(R, wctx, leader, S, reinterpret_cast<uint64_t>(&p.mapA[s]),
                                  reinterpret_cast<uint64_t>(&p.mapB[s]), kb0, kb1, row0, ncol0);
      }
      if (leader) claim = claim_ahead ? next : static_cast<int>(gridDim.x >> 1) + atomicAdd(sched, 1);
    }
    if (*abort_flag) {
      // Drain: the leader waits (bounded) until every stage it expected has
      // landed, which covers both CTAs' copies of those stages; the peer,
      // which cannot wait on the leader's barriers, lets a short fixed
      // interval pass for its own copies in flight.
      if (leader) {
        for (int s = 0; s < STAGES2; ++s) {
          if (!((R.pend_valid >> s) & 1u)) continue;
          const unsigned long long t0 = global_ns();
          while (!mbar_try_wait(full_bar(s), (R.pend_phase >> s) & 1u)) {
            if (global_ns() - t0 > p.wait_limit_ns) break;
          }
        }
      } else {
        const unsigned long long t0 = global_ns();
        while (global_ns() - t0 < 200000ull) __nanosleep(1000);
      }
    }
  } else if (warp == 1 && lane == 0 && leader) {
    // ------------------------- leader: pair MMA issuer -------------------------
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    bool issued_any = false;
    for (int lt = 0; ok; ++lt) {
      int tile;
      TileCoord tc;
      if (!take_tile(lt, tile, tc)) break;
      release_tile(lt);
      if (tile < 0) break;
      const GemmGroup& G = p.grp[tc.g];
      const int buf = lt & 1;
      const uint32_t tphase = static_cast<uint32_t>(lt >> 1) & 1u;
      if (!wait2(tempty_bar(buf), tphase ^ 1u, wctx)) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * BN);
      const int seg_begin = G.seg_begin, seg_end = G.seg_end;
      uint32_t acc = 0;
      for (int s = seg_begin; ok && s < seg_end; ++s) {
        const TcSeg S = p.seg[s];
        int kb0, kb1;
        tile_kb_range<BM2, ATTN>(G, S.K, tc.m0, tc.n0, kb0, kb1);
        const uint32_t idesc = idesc_bf16_m256(S.a_mn, S.b_mn, S.n_mma);
        const uint64_t a_desc0 = sdesc(tiles_base, S.a_mn ? MN_BOX_BYTES : 16, 1024);
        const uint64_t b_desc0 = sdesc(tiles_base + A_TILE_BYTES, S.b_mn ? MN_BOX_BYTES : 16, 1024);
        const uint32_t a_step = S.a_mn ? (2048 >> 4) : (32 >> 4);
        const uint32_t b_step = S.b_mn ? (2048 >> 4) : (32 >> 4);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!wait2(full_bar(stage), phase, wctx)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t off = static_cast<uint32_t>(stage * STAGE2_BYTES) >> 4;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            mma_bf16_pair(d_tmem, a_desc0 + off + kk * a_step, b_desc0 + off + kk * b_step, idesc, acc);
            acc = 1;
          }
          issued_any = true;
          mma_commit_pair(empty_bar(stage));
          if (++stage == STAGES2) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) break;
      mma_commit_pair(tfull_bar(buf));
    }
    if (*abort_flag && issued_any) {
      mma_commit_pair(drain_bar, 0x1);  // this CTA only
      const unsigned long long t0 = global_ns();
      while (!mbar_try_wait(drain_bar, 0)) {
        if (global_ns() - t0 > p.wait_limit_ns) break;
      }
    }
  } else if (warp >= 2) {
    // ---------------------------- epilogue (both CTAs) ----------------------------
    const int quarter = warp & 3;
    constexpr int cpw = BN / (32 * EPI_PARTS);  // 32-column chunks per warp
    const int c_begin = ((warp - 2) >> 2) * cpw;
    uint4* epi_stage = reinterpret_cast<uint4*>(smem + STAGES2 * STAGE2_BYTES + BAR_BYTES +
                                                (warp - 2) * EPI_WARP_BYTES);
    const uint32_t tempty_leader0 = map_to_rank(tempty_bar(0), 0);
    const uint32_t tempty_leader1 = map_to_rank(tempty_bar(1), 0);
    AuxLoad ax{smem_addr(aux_bars + (warp - 2)), 0u, abort_flag, p.err, p.wait_limit_ns};
    for (int lt = 0;; ++lt) {
      int tile;
      TileCoord tc;
      if (!take_tile(lt, tile, tc)) break;
      __syncwarp();
      if (lane == 0) release_tile(lt);
      if (tile < 0) break;
      const GemmGroup& G = p.grp[tc.g];
      const int buf = lt & 1;
      const uint32_t tphase = static_cast<uint32_t>(lt >> 1) & 1u;
      prefetch_bias(G, tc.n0 + c_begin * 32, lane);
      if (!wait2(tfull_bar(buf), tphase, wctx)) break;
      tc_fence_after();
      const int row0 = tc.m0 + 128 * static_cast<int>(rank) + quarter * 32;
      const uint32_t taddr =
          tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(buf * BN);
      const bool empty = tile_empty<BM2, ATTN>(p, G, tc.m0, tc.n0);
      if (G.epi == EPI_CE_FWD) ce_fwd_epilogue_warp<ATTN>(G, lane, row0, tc.n0, c_begin, cpw, taddr);
      if (ATTN && G.epi == EPI_SMAX_PARTS)
        smax_parts_epilogue_warp(G, p.mapO, epi_stage, lane, row0, tc.n0, c_begin, cpw, taddr);
      for (int c = c_begin; G.epi != EPI_CE_FWD && !(ATTN && G.epi == EPI_SMAX_PARTS) && c < c_begin + cpw;
           ++c) {
        const int n = tc.n0 + c * 32;
        if (n >= G.N) break;  // warp-uniform
        uint32_t rr[32];
        float v[32];
        if (empty) {
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = 0.f;
        } else {
          tmem_ld32(taddr + static_cast<uint32_t>(c * 32), rr);
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(rr[j]);
        }
        epilogue_chunk<ATTN>(G, p.mapO, epi_stage, ax, lane, row0, n, v);
      }
      tc_fence_before();
      if (G.prod_row >= 0 || G.prod_col >= 0) {
        if (lane == 0) {
          asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
          asm volatile("fence.proxy.async.global;" ::: "memory");
        }
        __threadfence();
        __syncwarp();
        if (lane == 0) {
          if (G.prod_row >= 0) atomicAdd(dep + G.prod_row + (tc.m0 + 128 * static_cast<int>(rank)) / BM, 1);
          if (G.prod_col >= 0) atomicAdd(dep + G.prod_col + tc.n0 / BN, 1);
        }
      }
      __syncwarp();
      if (lane == 0) {
        if (leader) mbar_arrive(tempty_bar(buf));
        else mbar_arrive_remote(buf ? tempty_leader1 : tempty_leader0);
      }
    }
  }

  // every bulk tensor store of the epilogue has finished before the CTA exits
  if (warp >= 2 && lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // no CTA touches the other's shared memory after this
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(TMEM_COLS)
                 : "memory");
  }
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(sched + 1, 1) == static_cast<int>(gridDim.x) - 1) {
      for (int c = 0; c < p.num_counters; ++c) atomicExch(dep + c, 0);
      atomicExch(sched, 0);
      atomicExch(sched + 1, 0);
    }
  }
}

// One-time set-up per device: the kernels' shared-memory limit is an
// attribute of each device's copy of the kernel, and the pair grid is sized
// by that device's occupancy.  Guarded so that threads making their first
// calls at the same time set it up once.
struct LaunchSetup {
  std::once_flag once;
  cudaError_t err = cudaSuccess;
  int max_clusters = 0;
};
constexpr int kSetupDevices = 64;
LaunchSetup g_setup[kSetupDevices];

cudaError_t setup_device(LaunchSetup& st, int num_sms) {
  cudaError_t e = cudaFuncSetAttribute(tc_gemm_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       SMEM_BYTES);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(tc_gemm_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(tc_gemm_pair_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             SMEM2_BYTES);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(tc_gemm_pair_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             SMEM2_BYTES);
  if (e != cudaSuccess) return e;
  // Every cluster of the persistent grid must be resident at once (tiles
  // may wait on tiles other clusters hold), so size the grid by occupancy.
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(2 * (num_sms / 2), 1, 1);
  cfg.blockDim = dim3(NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = SMEM2_BYTES;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(&st.max_clusters, tc_gemm_pair_kernel<false>, &cfg);
}

}  // namespace

cudaError_t launch_tc_gemm(const TcGemmParams& p_in, int num_sms, cudaStream_t s) {
  static std::atomic<unsigned> slot_seq{0};  // launch slots rotate across all host threads
  int dev = 0;
  cudaError_t de = cudaGetDevice(&dev);
  if (de != cudaSuccess) return de;
  if (dev < 0 || dev >= kSetupDevices) return cudaErrorInvalidDevice;
  LaunchSetup& st = g_setup[dev];
  std::call_once(st.once, [&] { st.err = setup_device(st, num_sms); });
  if (st.err != cudaSuccess) return st.err;
  const int max_clusters = st.max_clusters;
  if (p_in.total_tiles <= 0) return cudaSuccess;
  TcGemmParams& p = const_cast<TcGemmParams&>(p_in);
  p.sched_slot = static_cast<int>(slot_seq.fetch_add(1) % kSchedSlots);
  if (p.pair) {
    int clusters = max_clusters < num_sms / 2 ? max_clusters : num_sms / 2;
    if (clusters > p.total_tiles) clusters = p.total_tiles;
    if (clusters < 1) return cudaErrorInvalidConfiguration;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = pdl_on() ? 1 : 0;
    cfg.gridDim = dim3(2 * clusters, 1, 1);
    cfg.blockDim = dim3(NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = SMEM2_BYTES;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    cudaError_t e = p.attn ? cudaLaunchKernelEx(&cfg, tc_gemm_pair_kernel<true>, p)
                           : cudaLaunchKernelEx(&cfg, tc_gemm_pair_kernel<false>, p);
    count_launches(1);
    return e != cudaSuccess ? e : cudaGetLastError();
  }
  const int grid = p.total_tiles < num_sms ? p.total_tiles : num_sms;
  const cudaError_t e = p.attn ? launch_k(tc_gemm_kernel<true>, grid, NUM_THREADS, SMEM_BYTES, s, p)
                               : launch_k(tc_gemm_kernel<false>, grid, NUM_THREADS, SMEM_BYTES, s, p);
  count_launches(1);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace tp
