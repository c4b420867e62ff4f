// Fused row-parallel GEMM + partial channel-reduce on the 5th-generation tensor
// core (sm_103a): TMA tile loads, tcgen05.mma with accumulators in TMEM, and an
// epilogue that writes the t rank outputs.
//
// "Tensor-Parallelism with Partially Synchronized Activations", Introduction,
// partial channel-reduce paragraph: after the row-parallel layer (Y_r = X_r W_r,
// K split t ways), channels in S are summed over the ranks and every rank gets
// the sum; the other channels keep each rank's own partial result.
//
// One persistent CTA per SM walks output tiles of 128 rows x 256 channels (or
// 192 channels where h is a multiple of 192; CTA pairs take 256-row tiles).
// Every tile streams the same k-blocks (shard 0's K slice, then shard 1's, ...),
// so all tiles cost the same MMA work; what differs is where results go:
//   FULL_S tile (every channel in S): one accumulation over all of K (that is
//     X W[:, tile] = sum_r Y_r), written to all t outputs;
//   NO_S tile (no channel in S): a fresh accumulation per shard, written to that
//     rank's output after each shard;
//   MIXED tile: shard r accumulates into TMEM buffer (r mod 2).  After each
//     shard the epilogue writes the buffer to Y_r and zeroes the non-S columns,
//     so the S columns keep summing (even shards in one buffer, odd shards in
//     the other); after the last shard the two buffers' S columns are added and
//     written to every rank.
// Two fp32 accumulators (256 TMEM columns apart; all 512 columns allocated)
// alternate, so the epilogue of one accumulation overlaps the MMAs of the next.
//
// Compact outputs (a contiguous S of a multiple of 64 channels): the S channels
// are written once, to YS [N, |S|], and rank r's other channels to YN[r]
// [N, h - |S|].  Every 64-channel chunk is then all in S or all outside it: a
// FULL_S tile stores each chunk once, a NO_S tile at its column minus |S|, and a
// MIXED tile skips its S chunks until the last shard, which stores their sums to
// YS (no per-rank stores of the sums).
//
// Warp roles: warp 0 lane 0 issues TMA loads into a 4-stage ring, warp 1 lane 0
// issues the MMAs (warp 1 also owns the TMEM allocation), warps 2..5 drain TMEM
// (each warp reads the 32 TMEM lanes its rank within the warp quad may access).
// The K slices are fetched through 3-D tensor maps (k within shard, shard, row),
// so a shard whose width is not a multiple of 64 reads zeros past its end instead
// of the next shard's columns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdlib>
#include <cstring>

#include "caat_internal.h"
#include "tc_ptx.cuh"

namespace caat {

__device__ int g_caat_dev_error;

caat_status read_and_clear_bwd_error();
caat_status read_and_clear_skinny_error();

caat_status read_and_clear_device_error()
{
    const caat_status sb = read_and_clear_bwd_error();
    if (sb != CAAT_OK) return sb;
    const caat_status ss = read_and_clear_skinny_error();
    if (ss != CAAT_OK) return ss;
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_caat_dev_error, sizeof(int)) != cudaSuccess) return CAAT_ERR_CUDA;
    if (v != 0) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(g_caat_dev_error, &zero, sizeof(int)) != cudaSuccess) return CAAT_ERR_CUDA;
        return (caat_status)v;
    }
    return CAAT_OK;
}

// The tensor-map encoder is a driver-API function; it is looked up through the
// runtime so the library does not link libcuda itself.
static PFN_cuTensorMapEncodeTiled_v12000 lookup_encoder()
{
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return nullptr;
    return (PFN_cuTensorMapEncodeTiled_v12000)f;
}

// bf16 (or fp32) tensor map with the 128-byte swizzle, zero fill out of bounds.
// dims[0] is the contiguous dimension; strides_bytes[i] is the stride of dims[i+1].
bool encode_tmap(CUtensorMap *tm, const void *base, int rank, const uint64_t *dims,
                 const uint64_t *strides_bytes, const uint32_t *box, bool f32)
{
    static const PFN_cuTensorMapEncodeTiled_v12000 encode = lookup_encoder();   // thread-safe init
    if (encode == nullptr || rank < 1 || rank > 5) return false;
    cuuint64_t d[5], st[4];
    cuuint32_t bx[5], es[5];
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        bx[i] = box[i];
        es[i] = 1;
        if (i + 1 < rank) st[i] = strides_bytes[i];
    }
    const CUresult r = encode(tm, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void *>(base),
                              d, st, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

namespace {

using namespace tc;

constexpr int BM = 128, BN = 256, BK = 64;
constexpr int A_BYTES = BM * BK * 2;
constexpr int NUM_THREADS = 192;
constexpr uint32_t TMEM_COLS = 512;
constexpr int MAX_H_TC = 32768;
constexpr int MAX_T_TC = 16;                 // rank outputs addressed through tensor maps
constexpr int STG_BYTES = 32 * 128;          // per epilogue warp: 32 rows x 64 bf16 channels
constexpr int MAX_STAGES = 8;
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;   // 2 s: far beyond any legitimate wait

// failure-path test hooks (caat_debug_set_wait): the wait limit and the injected
// failure the next launches take
std::atomic<uint64_t> g_wait_ns{WAIT_LIMIT_NS};
std::atomic<int> g_inject{CAAT_INJECT_NONE};

// Per mode: PAIR = false, one CTA computes a 128 x 256 tile (4 stages of X 128 x 64
// + W 256 x 64, one staging buffer per epilogue warp); PAIR = true, a CTA pair
// computes a 256 x 256 tile with one cta_group::2 MMA (5 stages of X 128 x 64 +
// W 128 x 64 per CTA: each CTA holds half the rows of X and half the channels of
// W, which cuts the shared-memory operand traffic per SM by a third; two staging
// buffers per epilogue warp so a bulk store can drain while the next is staged).
// Ring depth of the pair mode and the staging buffers per epilogue warp of its
// 256-wide tiles (compile-time tuning; shared memory holds stages x 32 KB plus
// 4 x NBUF x 4 KB of staging).
#ifndef CAAT_FWD_PAIR_STAGES
#define CAAT_FWD_PAIR_STAGES 6
#endif
#ifndef CAAT_FWD_PAIR_NBUF256
#define CAAT_FWD_PAIR_NBUF256 1
#endif
// DEEP (single-CTA 192-wide tiles only): 5 ring stages of 40 KB and one staging
// buffer per epilogue warp instead of 4 stages and two.  Shards of 4 or more
// k-blocks are fed faster (130M down-proj, k_t = 384: 49.3 -> 46.6 us); shorter
// shards are bound by their per-shard epilogue, which the second buffer helps
// (130M out-proj, k_t = 96: 33.5 against 35.2 us).
// STG2 (256-wide tiles): two staging buffers per epilogue warp instead of one,
// taken when the S bitmap of the call leaves room for them next to the ring (6
// stages of 32 KB for CTA pairs, 4 of 48 KB for single CTAs; h up to about
// 15,000 channels).  A bulk store then drains one buffer while the next chunk
// fills the other (7B prefill out-proj: 114 -> 111 us).
template <int CLN, int BNT, bool DEEP = false, bool STG2 = false>
struct Cfg {
    static constexpr bool PAIR = CLN > 1;
    static constexpr int STAGES = PAIR ? CAAT_FWD_PAIR_STAGES : (BNT < 256 && DEEP ? 5 : 4);
    // staging buffers per epilogue warp: several (bulk stores drain the earlier
    // ones while the next chunk fills one) where shared memory allows
    static constexpr int NBUF = BNT < 256 ? (DEEP ? 1 : 2) : (STG2 ? 2 : (PAIR ? CAAT_FWD_PAIR_NBUF256 : 1));
    static constexpr int B_ROWS = PAIR ? BNT / 2 : BNT;        // W rows (channels) per CTA per stage
    static constexpr int B_BYTES = B_ROWS * BK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr uint32_t TX_BYTES = (PAIR ? 2 : 1) * STAGE_BYTES;   // landing per stage (leader)
    static constexpr uint32_t IDESC = idesc_bf16_f32(PAIR ? 2 * BM : BM, BNT);
};

enum { FULL_S = 0, NO_S = 1, MIXED = 2 };

struct SmemCtl {
    uint64_t full[MAX_STAGES];
    uint64_t empty[MAX_STAGES];
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint32_t tmem_base;
    int abort;
    // followed in shared memory by the S bitmap: ceil(h / 32) words and two
    // zero words after them (the epilogue reads a chunk's two words at once)
};

// shared memory of a mode without the S bitmap (which takes ceil(h / 32) words more)
template <int CLN, int BNT, bool DEEP, bool STG2>
constexpr size_t smem_bytes()
{
    using C = Cfg<CLN, BNT, DEEP, STG2>;
    static_assert(C::STAGES <= MAX_STAGES, "ring deeper than the barrier arrays");
    return 1024 + (size_t)C::STAGES * C::STAGE_BYTES + 4 * C::NBUF * STG_BYTES +
           sizeof(SmemCtl);
}
constexpr size_t bitmap_bytes(int64_t h) { return (size_t)((h + 31) / 32 + 2) * 4; }

struct YMaps {
    CUtensorMap m[MAX_T_TC];   // rank r's output [N, h] (compact: [N, h - |S|]), box 64 channels x 32 rows
    CUtensorMap s;             // compact outputs: the S channels [N, |S|], same box
};

constexpr int MAX_NB = (MAX_H_TC + 191) / 192;   // channel blocks at the narrowest tile

struct FwdParams {
    MutPtrs Y;
    int64_t ldy;
    int64_t N, h;
    int t, nkb, num_m, num_n;
    int mmajor;         // work units ordered row-block-major (else channel-block-major)
    // Balanced schedule (contiguous S, some channel blocks outside S): the first
    // n_whole entries of nbl are the channel blocks whose tiles run whole (FULL_S,
    // MIXED), the rest the NO_S blocks, whose tiles are cut into one piece per
    // shard.  balanced == 0: every tile runs whole, in unit order.
    int balanced;
    int n_whole;
    int wgt;            // pieces a whole tile's time is worth (1 .. t): the light workers' extra share
    uint8_t nbl[MAX_NB];
    const int32_t *sel;
    int64_t n_sel;
    uint64_t wait_ns;   // limit of every mbarrier wait
    int inject;         // CAAT_INJECT_SKIP_LOADS: the producer issues nothing
};

__device__ __forceinline__ void fail(volatile int *abort)
{
    *abort = 1;
    atomicExch(&g_caat_dev_error, (int)CAAT_ERR_TIMEOUT);
}

// ------------------------------------------------------------ work schedule
// Workers are CTAs (CTA pairs in the pair mode), g = 0 .. G-1.  Every shard of
// every tile costs the same MMA work, so a tile that runs whole costs t shards
// and a NO_S tile can be cut into t independent one-shard pieces (each writes
// only its own rank's output).  Whole tiles go round-robin to the workers (in
// unit order).  The pieces are numbered shard-major (all tiles' shard 0, then
// shard 1, ...) and also dealt round-robin, so at any moment the workers run
// neighbouring tiles at the same shard and share their X and W blocks in L2.
// When the whole tiles leave some workers one tile short (the "light" workers),
// the first light x t pieces go to those alone, which evens out the load.
struct Work {
    int mg, nb;    // row group (CLN row blocks) and channel block
    int r0, r1;    // shards [r0, r1) of the tile
    int piece;     // 1: a one-shard piece of a NO_S tile
};

struct Cursor {
    int i;            // next whole unit
    int j, step, end; // next piece, stride, end of the current phase
    int phase;        // 0: pieces for the light workers, 1: pieces for all, 2: done
    int wleft;        // whole units still to come (interleaved order)
    int batch, inb;   // pieces between two whole units, pieces of the current run
};

__device__ __forceinline__ void cursor_init(Cursor &c, const FwdParams &p, int g, int G, int num_mg)
{
    c.i = g;
    c.phase = 2;
    c.wleft = c.batch = c.inb = 0;
    if (!p.balanced) return;
    const int nW = num_mg * p.n_whole;
    const int rem = nW % G;
    const int light = rem > 0 ? G - rem : 0;
    const int P = num_mg * (p.num_n - p.n_whole) * p.t;
    const int A = min(P, light * p.wgt);
    int q = 0;    // this worker's pieces
    if (light > 0 && g >= rem && g - rem < A) {
        c.phase = 0;
        c.j = g - rem;
        c.step = light;
        c.end = A;
        q = (A - c.j + light - 1) / light;
    } else {
        c.phase = 1;
        c.j = A + g;
        c.step = G;
        c.end = P;
    }
    if (A + g < P) q += (P - (A + g) + G - 1) / G;
    c.wleft = g < nW ? (nW - 1 - g) / G + 1 : 0;
    // interleaved order: the pieces in wleft + 1 equal runs around the whole units
    c.batch = (q + c.wleft) / (c.wleft + 1);
}

__device__ __forceinline__ bool next_piece(Cursor &c, const FwdParams &p, int g, int G, int num_mg, Work &w)
{
    if (c.phase == 0 && c.j >= c.end) {
        // the light workers' share is done: continue with the pieces dealt to all
        c.phase = 1;
        c.j = c.end + g;
        c.step = G;
        c.end = num_mg * (p.num_n - p.n_whole) * p.t;
    }
    if (c.phase == 2 || c.j >= c.end) return false;
    const int nsb = p.num_n - p.n_whole;
    const int ntiles = num_mg * nsb;
    const int r = c.j / ntiles, tile = c.j - r * ntiles;
    w.r0 = r;
    w.r1 = r + 1;
    w.mg = p.mmajor ? tile / nsb : tile % num_mg;
    w.nb = p.nbl[p.n_whole + (p.mmajor ? tile % nsb : tile / num_mg)];
    w.piece = 1;
    c.j += c.step;
    return true;
}

__device__ __forceinline__ bool next_whole(Cursor &c, const FwdParams &p, int G, int num_mg, Work &w)
{
    const int nW = num_mg * p.n_whole;
    if (c.i >= nW) return false;
    const int i = c.i;
    c.i += G;
    w.mg = p.mmajor ? i / p.n_whole : i % num_mg;
    w.nb = p.nbl[p.mmajor ? i % p.n_whole : i / num_mg];
    w.r0 = 0;
    w.r1 = p.t;
    w.piece = 0;
    return true;
}

// The next work item of worker g.  balanced == 1: the whole units first, then the
// pieces; balanced == 2: the pieces in equal runs before, between and after the
// whole units, which spreads the pieces' output writes over the whole kernel.
__device__ __forceinline__ bool next_work(Cursor &c, const FwdParams &p, int g, int G, int num_mg, Work &w)
{
    if (!p.balanced) {
        if (c.i >= num_mg * p.num_n) return false;
        const int u = c.i;
        c.i += G;
        w.mg = p.mmajor ? u / p.num_n : u % num_mg;
        w.nb = p.mmajor ? u % p.num_n : u / num_mg;
        w.r0 = 0;
        w.r1 = p.t;
        w.piece = 0;
        return true;
    }
    if (p.balanced == 1) {
        if (next_whole(c, p, G, num_mg, w)) return true;
        return next_piece(c, p, g, G, num_mg, w);
    }
    if (c.inb < c.batch && next_piece(c, p, g, G, num_mg, w)) {
        ++c.inb;
        return true;
    }
    if (c.wleft > 0 && next_whole(c, p, G, num_mg, w)) {
        --c.wleft;
        c.inb = 0;
        return true;
    }
    return next_piece(c, p, g, G, num_mg, w);
}

template <int BNT>
__device__ __forceinline__ int tile_class(const uint32_t *bm, int64_t n0, int64_t h, int t)
{
    if (t == 1) return FULL_S;
    bool any = false, all = true;
#pragma unroll
    for (int w = 0; w < BNT / 32; ++w) {
        const int64_t c = n0 + 32 * w;
        if (c < h) {
            const int64_t nv = h - c < 32 ? h - c : 32;
            const uint32_t valid = nv == 32 ? 0xffffffffu : ((1u << nv) - 1u);
            const uint32_t bits = bm[c >> 5] & valid;
            any = any || bits != 0u;
            all = all && bits == valid;
        }
    }
    return all ? FULL_S : (any ? MIXED : NO_S);
}

__device__ __forceinline__ uint32_t pack_bf16x2(uint32_t lo_f32, uint32_t hi_f32)
{
    const __nv_bfloat162 v = __floats2bfloat162_rn(__uint_as_float(lo_f32), __uint_as_float(hi_f32));
    return *reinterpret_cast<const uint32_t *>(&v);
}

// CLN = CTAs per cluster: 1 (one CTA per tile) or 2 (a CTA pair).  Each CTA
// fetches its own X and W tiles from this GPU's memory; no load is multicast.
// COMPACT: the compact outputs (ymaps.s and the shifted ymaps.m), a separate
// instantiation so that the plain epilogue carries none of its branches.
template <int CLN, int BNT, bool DEEP, bool STG2, bool COMPACT>
__global__ void __launch_bounds__(NUM_THREADS, 1)
rowpar_fwd_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                     const __grid_constant__ YMaps ymaps, const FwdParams p)
{
    using C = Cfg<CLN, BNT, DEEP, STG2>;
    constexpr bool PAIR = C::PAIR;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t *smA = base;
    uint8_t *smB = base + C::STAGES * A_BYTES;
    uint8_t *staging = base + C::STAGES * C::STAGE_BYTES;
    SmemCtl *ctl = (SmemCtl *)(staging + 4 * C::NBUF * STG_BYTES);
    uint32_t *bitmap = reinterpret_cast<uint32_t *>(ctl + 1);
    volatile int *abort = &ctl->abort;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t words = (p.h + 31) >> 5;
    const uint32_t crank = PAIR ? cluster_ctarank() : 0u;
    const uint32_t leader = crank & ~1u;                    // even CTA of this CTA's pair
    const bool is_leader = crank == leader;

    for (int64_t w = tid; w < words + 2; w += NUM_THREADS) bitmap[w] = 0u;
    if (tid == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(smem_u32(&ctl->full[s]), 1);
            mbar_init(smem_u32(&ctl->empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&ctl->acc_full[b]), 1);
            mbar_init(smem_u32(&ctl->acc_empty[b]), PAIR ? 256 : 128);
        }
        ctl->abort = 0;
        fence_mbar_init();
        prefetch_tmap(&tmX);
        prefetch_tmap(&tmW);
    }
    if (PAIR) cluster_sync();        // the peer's barriers exist before anything signals them
    else __syncthreads();
    if (warp == 1) {
        if (PAIR) {
            tmem_alloc_pair(smem_u32(&ctl->tmem_base), TMEM_COLS);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(smem_u32(&ctl->tmem_base), TMEM_COLS);
            tmem_relinquish();
        }
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = ctl->tmem_base;
    // Launched as a programmatic dependent, this grid may have started while the
    // previous one in the stream was still running: nothing above touched global
    // memory (the tensor maps are launch parameters).  Wait for it before the
    // first global read or write, then let the next grid start its own setup.
    griddep_wait();
    griddep_launch_dependents();
    if (warp != 0) {
        // The channel bitmap of S, built by the MMA and epilogue warps while the
        // producer already streams the first stages (it needs no bitmap): every
        // index of S is read once, eight independent loads per thread in flight.
        const int e = tid - 32;
        constexpr int NB = NUM_THREADS - 32;
        if (p.sel == nullptr) {      // S = {0, ..., n_sel-1}
            for (int64_t w = e; w < words; w += NB) {
                const int64_t lo = w * 32;
                bitmap[w] = p.n_sel >= lo + 32 ? 0xffffffffu
                               : (p.n_sel <= lo ? 0u : ((1u << (p.n_sel - lo)) - 1u));
            }
        } else {
            for (int64_t i0 = e; i0 < p.n_sel; i0 += (int64_t)NB * 8) {
                int32_t v[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) v[u] = i0 + NB * u < p.n_sel ? __ldg(p.sel + i0 + NB * u) : -1;
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    if (v[u] >= 0 && v[u] < p.h) atomicOr(&bitmap[v[u] >> 5], 1u << (v[u] & 31));
            }
        }
        asm volatile("bar.sync 1, %0;" ::"n"(NB) : "memory");   // warps 1..5
    }

    // work items: (group of CLN row blocks, channel block, shard range); the CTAs
    // of a cluster take the row blocks of a group
    const int worker = blockIdx.x / CLN;
    const int nworkers = gridDim.x / CLN;
    const int num_mg = (p.num_m + CLN - 1) / CLN;

    if (warp == 0) {
        // ---------------------------------------------------- TMA producer
        if (lane == 0 && p.inject != CAAT_INJECT_SKIP_LOADS) {
            int stage = 0;
            uint32_t ph = 0;
            Cursor cur;
            cursor_init(cur, p, worker, nworkers, num_mg);
            Work wk;
            while (next_work(cur, p, worker, nworkers, num_mg, wk)) {
                const int mb = wk.mg * CLN + (int)crank;
                const int nb = wk.nb;
                for (int r = wk.r0; r < wk.r1; ++r) {
                    for (int kb = 0; kb < p.nkb; ++kb) {
                        if (!mbar_wait(smem_u32(&ctl->empty[stage]), ph ^ 1u, abort, p.wait_ns)) {
                            fail(abort);
                            goto done;
                        }
                        const uint32_t fb = smem_u32(&ctl->full[stage]);
                        if (PAIR) {
                            // both CTAs' halves land on the pair leader's barrier
                            const uint32_t fl = map_to_cta(fb, leader);
                            if (is_leader) mbar_arrive_expect_tx(fb, C::TX_BYTES);
                            tma_load_3d_pair(smem_u32(smA + stage * A_BYTES), &tmX, fl, kb * BK, r, mb * BM);
                            tma_load_3d_pair(smem_u32(smB + stage * C::B_BYTES), &tmW, fl, kb * BK, r,
                                             nb * BNT + (int)crank * C::B_ROWS);
                        } else {
                            mbar_arrive_expect_tx(fb, C::TX_BYTES);
                            tma_load_3d(smem_u32(smA + stage * A_BYTES), &tmX, fb, kb * BK, r, mb * BM);
                            tma_load_3d(smem_u32(smB + stage * C::B_BYTES), &tmW, fb, kb * BK, r, nb * BNT);
                        }
                        if (++stage == C::STAGES) { stage = 0; ph ^= 1u; }
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------ MMA issuer
        if (lane == 0 && is_leader) {
            const uint16_t pair_mask = (uint16_t)(3u << leader);
            int stage = 0;
            uint32_t ph = 0, au = 0;
            Cursor cur;
            cursor_init(cur, p, worker, nworkers, num_mg);
            Work wk;
            while (next_work(cur, p, worker, nworkers, num_mg, wk)) {
                const int nb = wk.nb;
                const int cls = wk.piece ? (int)NO_S : tile_class<BNT>(bitmap, (int64_t)nb * BNT, p.h, p.t);
                for (int r = wk.r0; r < wk.r1; ++r) {
                    const bool starts = cls != FULL_S || r == 0;
                    const bool ends = cls != FULL_S || r == p.t - 1;
                    const uint32_t b = au & 1u;
                    if (starts) {
                        if (!mbar_wait(smem_u32(&ctl->acc_empty[b]), ((au >> 1) & 1u) ^ 1u, abort,
                                       p.wait_ns)) {
                            fail(abort);
                            goto done;
                        }
                        fence_after_sync();
                    }
                    const bool fresh = cls == FULL_S ? r == 0 : (cls == NO_S ? true : r < 2);
                    const uint32_t d = tmem + b * 256u;
                    for (int kb = 0; kb < p.nkb; ++kb) {
                        if (!mbar_wait(smem_u32(&ctl->full[stage]), ph, abort, p.wait_ns)) {
                            fail(abort);
                            goto done;
                        }
                        fence_after_sync();
                        const uint32_t a0 = smem_u32(smA + stage * A_BYTES);
                        const uint32_t b0 = smem_u32(smB + stage * C::B_BYTES);
#pragma unroll
                        for (int k = 0; k < BK / 16; ++k) {
                            const uint64_t ad = desc_kmajor_sw128(a0 + 32u * k);
                            const uint64_t bd = desc_kmajor_sw128(b0 + 32u * k);
                            const uint32_t acc = (fresh && kb == 0 && k == 0) ? 0u : 1u;
                            if (PAIR) mma_f16_pair(d, ad, bd, C::IDESC, acc);
                            else mma_f16(d, ad, bd, C::IDESC, acc);
                        }
                        if (PAIR) mma_commit_pair_mc(smem_u32(&ctl->empty[stage]), pair_mask);
                        else mma_commit(smem_u32(&ctl->empty[stage]));
                        if (++stage == C::STAGES) { stage = 0; ph ^= 1u; }
                    }
                    if (ends) {
                        if (PAIR) mma_commit_pair_mc(smem_u32(&ctl->acc_full[b]), pair_mask);
                        else mma_commit(smem_u32(&ctl->acc_full[b]));
                        ++au;
                    }
                }
            }
        }
    } else {
        // -------------------------------------------------------- epilogue
        const int q = warp & 3;                         // TMEM lane quarter of this warp
        const uint32_t lane_off = (uint32_t)(32 * q) << 16;
        uint32_t au = 0;
        int sbuf = 0;                                   // staging buffer the next chunk fills
        Cursor cur;
        cursor_init(cur, p, worker, nworkers, num_mg);
        Work wk;
        while (next_work(cur, p, worker, nworkers, num_mg, wk)) {
            const int mb = wk.mg * CLN + (int)crank;
            const int nb = wk.nb;
            const int64_t n0 = (int64_t)nb * BNT;
            const int cls = wk.piece ? (int)NO_S : tile_class<BNT>(bitmap, n0, p.h, p.t);
            for (int r = wk.r0; r < wk.r1; ++r) {
                if (cls == FULL_S && r != p.t - 1) continue;
                const uint32_t b = au & 1u;
                bool ok = mbar_wait(smem_u32(&ctl->acc_full[b]), (au >> 1) & 1u, abort, p.wait_ns);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) {
                    fail(abort);
                    goto done;
                }
                fence_after_sync();
                const uint32_t tb = tmem + lane_off + b * 256u;
                const uint32_t tb_other = tmem + lane_off + (b ^ 1u) * 256u;
                const bool final_mixed = cls == MIXED && r == p.t - 1;
                const bool zero_nons = cls == MIXED && r <= p.t - 3;
                const int y = mb * BM + 32 * q;
                uint8_t *stg = staging + q * C::NBUF * STG_BYTES;   // this warp's first buffer
                if (!final_mixed) {
                    // Stage 32 rows x 64 channels in shared memory (128-byte swizzle:
                    // 16-byte chunk j of row i sits at chunk j ^ (i mod 8)), then one
                    // bulk tensor store per destination rank -- the same staged tile
                    // serves all t ranks of a FULL_S tile.  A MIXED shard before the
                    // last writes its partials whole: its S channels are rewritten
                    // with the sum at the end.
#pragma unroll 1
                    for (int c64 = 0; c64 < BNT / 64; ++c64) {
                        const int64_t c0 = n0 + 64 * c64;
                        if (c0 >= p.h) break;             // same for the whole warp
                        uint32_t v0[32], v1[32];
                        tmem_ld32x2(tb + 64u * c64, tb + 64u * c64 + 32u, v0, v1);
                        uint32_t w[32];
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            w[i] = pack_bf16x2(v0[2 * i], v0[2 * i + 1]);
                            w[16 + i] = pack_bf16x2(v1[2 * i], v1[2 * i + 1]);
                        }
                        if (zero_nons) {
                            // keep the S channels accumulating, clear the others
                            const uint32_t m0 = bitmap[c0 >> 5], m1 = bitmap[(c0 >> 5) + 1];
#pragma unroll
                            for (int j = 0; j < 32; ++j) {
                                v0[j] = ((m0 >> j) & 1u) ? v0[j] : 0u;
                                v1[j] = ((m1 >> j) & 1u) ? v1[j] : 0u;
                            }
                            tmem_st32(tb + 64u * c64, v0);
                            tmem_st32(tb + 64u * c64 + 32u, v1);
                        }
                        // compact outputs: a MIXED shard's S chunks are still summing
                        if (COMPACT && cls == MIXED && c0 < p.n_sel) continue;
                        // the buffer to fill: every earlier bulk group but the last has
                        // read its staging (the last one read the other buffer)
                        uint8_t *stgc = stg + sbuf * STG_BYTES;
                        const uint32_t stgc_a = smem_u32(stgc);
                        if (lane == 0) {
                            bulk_wait_read_n<C::NBUF - 1>();
                        }
                        __syncwarp();
                        uint4 *rowp = reinterpret_cast<uint4 *>(stgc + lane * 128);
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            rowp[j ^ (lane & 7)] = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (y < p.N) {                     // same for the whole warp
                            if (lane == 0) {
                                if (COMPACT && c0 < p.n_sel) {
                                    tma_store_2d(&ymaps.s, stgc_a, (int)c0, y);     // the sum, once
                                } else {
                                    const int xc = COMPACT ? (int)(c0 - p.n_sel) : (int)c0;
                                    if (cls == FULL_S) {
                                        for (int rr = 0; rr < p.t; ++rr) tma_store_2d(&ymaps.m[rr], stgc_a, xc, y);
                                    } else {
                                        tma_store_2d(&ymaps.m[r], stgc_a, xc, y);
                                    }
                                }
                                bulk_commit();
                            }
                            if (C::NBUF > 1) sbuf = sbuf + 1 == C::NBUF ? 0 : sbuf + 1;   // one bulk group per filled buffer
                        }
                    }
                } else {
                    const uint32_t stg_a = smem_u32(stg);
                    // Last shard of a MIXED tile: rank t-1's tile (S channels from
                    // the sum of both accumulators, the others its own) by bulk
                    // store; then the S sums into the other ranks' S channels with
                    // row-coalesced, per-lane masked stores, after this warp's
                    // earlier bulk stores to those rows have completed.
#pragma unroll 1
                    for (int c64 = 0; c64 < BNT / 64; ++c64) {
                        const int64_t c0 = n0 + 64 * c64;
                        if (c0 >= p.h) break;
                        const uint32_t m0 = bitmap[c0 >> 5], m1 = bitmap[(c0 >> 5) + 1];
                        uint32_t w[32], ws[32];
                        {
                            uint32_t v[32], u[32];
                            tmem_ld32x2(tb + 64u * c64, tb_other + 64u * c64, v, u);
#pragma unroll
                            for (int i = 0; i < 16; ++i) {
                                const float s0 = __uint_as_float(u[2 * i]) + __uint_as_float(v[2 * i]);
                                const float s1 = __uint_as_float(u[2 * i + 1]) + __uint_as_float(v[2 * i + 1]);
                                ws[i] = pack_bf16x2(__float_as_uint(s0), __float_as_uint(s1));
                                w[i] = pack_bf16x2(((m0 >> (2 * i)) & 1u) ? __float_as_uint(s0) : v[2 * i],
                                                   ((m0 >> (2 * i + 1)) & 1u) ? __float_as_uint(s1) : v[2 * i + 1]);
                            }
                            tmem_ld32x2(tb + 64u * c64 + 32u, tb_other + 64u * c64 + 32u, v, u);
#pragma unroll
                            for (int i = 0; i < 16; ++i) {
                                const float s0 = __uint_as_float(u[2 * i]) + __uint_as_float(v[2 * i]);
                                const float s1 = __uint_as_float(u[2 * i + 1]) + __uint_as_float(v[2 * i + 1]);
                                ws[16 + i] = pack_bf16x2(__float_as_uint(s0), __float_as_uint(s1));
                                w[16 + i] = pack_bf16x2(((m1 >> (2 * i)) & 1u) ? __float_as_uint(s0) : v[2 * i],
                                                        ((m1 >> (2 * i + 1)) & 1u) ? __float_as_uint(s1) : v[2 * i + 1]);
                            }
                        }
                        uint4 *rowp = reinterpret_cast<uint4 *>(stg + lane * 128);
                        if (COMPACT) {
                            // an S chunk: its sums, once, to YS; any other chunk: rank
                            // t-1's own partials (w, no S channel in it) to YN[t-1]
                            const bool sch = c0 < p.n_sel;
                            if (lane == 0) bulk_wait_read0();
                            __syncwarp();
#pragma unroll
                            for (int j = 0; j < 8; ++j)
                                rowp[j ^ (lane & 7)] = sch ? make_uint4(ws[4 * j], ws[4 * j + 1], ws[4 * j + 2], ws[4 * j + 3])
                                                           : make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
                            fence_proxy_async_smem();
                            __syncwarp();
                            if (lane == 0 && y < p.N) {
                                if (sch) tma_store_2d(&ymaps.s, stg_a, (int)c0, y);
                                else tma_store_2d(&ymaps.m[p.t - 1], stg_a, (int)(c0 - p.n_sel), y);
                                bulk_commit();
                            }
                            continue;
                        }
                        if (lane == 0) bulk_wait_read0();
                        __syncwarp();
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            rowp[j ^ (lane & 7)] = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0 && y < p.N) {
                            tma_store_2d(&ymaps.m[p.t - 1], stg_a, (int)c0, y);
                            bulk_commit();
                        }
                        // the sums, staged the same way, once the store above has read
                        // the staging; then every earlier bulk store of this warp (the
                        // shards' partials in these rows) must be complete before the
                        // generic stores below overwrite their S channels
                        if (lane == 0) {
                            bulk_wait0();
                            fence_proxy_async_global();
                        }
                        __syncwarp();
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            rowp[j ^ (lane & 7)] = make_uint4(ws[4 * j], ws[4 * j + 1], ws[4 * j + 2], ws[4 * j + 3]);
                        __syncwarp();
                        // lane l owns channel c0 + l (and c0 + 32 + l) of every row
                        const bool s_lo = (m0 >> lane) & 1u, s_hi = (m1 >> lane) & 1u;
                        const bool ok_lo = s_lo && c0 + lane < p.h, ok_hi = s_hi && c0 + 32 + lane < p.h;
                        if (__any_sync(0xffffffffu, ok_lo || ok_hi)) {
                            for (int i = 0; i < 32; ++i) {
                                const int64_t grow = (int64_t)y + i;
                                if (grow >= p.N) break;
                                const uint8_t *srow = stg + i * 128;
                                const uint16_t vlo = *reinterpret_cast<const uint16_t *>(
                                    srow + (((lane >> 3) ^ (i & 7)) << 4) + (lane & 7) * 2);
                                const uint16_t vhi = *reinterpret_cast<const uint16_t *>(
                                    srow + ((((lane + 32) >> 3) ^ (i & 7)) << 4) + (lane & 7) * 2);
                                for (int rr = 0; rr < p.t - 1; ++rr) {
                                    uint16_t *yrow = (uint16_t *)p.Y.p[rr] + grow * p.ldy + c0;
                                    if (ok_lo) yrow[lane] = vlo;
                                    if (ok_hi) yrow[32 + lane] = vhi;
                                }
                            }
                        }
                        __syncwarp();
                    }
                }
                fence_before_sync();
                // release the accumulator(s) to the MMA issuer (the pair leader's barrier)
                const uint32_t eb = smem_u32(&ctl->acc_empty[b]);
                const uint32_t eb2 = smem_u32(&ctl->acc_empty[b ^ 1u]);
                if (cls != MIXED || r <= p.t - 3 || final_mixed) {
                    if (PAIR) mbar_arrive_cluster(map_to_cta(eb, leader)); else mbar_arrive(eb);
                }
                if (final_mixed) {
                    if (PAIR) mbar_arrive_cluster(map_to_cta(eb2, leader)); else mbar_arrive(eb2);
                }
                ++au;
            }
        }
    }

done:
    if (warp >= 2 && lane == 0) bulk_wait0();   // bulk stores done before shared memory goes away
    fence_before_sync();
    __syncthreads();
    if (*abort) {
        // let copies and MMAs already in flight land before TMEM and shared
        // memory go away
        if (tid == 0) {
            const uint64_t t0 = globaltimer();
            while (globaltimer() - t0 < 2000000ull) { }
        }
        __syncthreads();
    }
    if (PAIR) cluster_sync();        // neither CTA leaves while its peer may still signal it
    if (warp == 1) {
        __syncwarp();
        fence_after_sync();
        if (PAIR) tmem_dealloc_pair(tmem, TMEM_COLS);
        else tmem_dealloc(tmem, TMEM_COLS);
    }
}

bool encode_3d(CUtensorMap *tm, const void *base, uint64_t d0, uint64_t d1, uint64_t d2,
               uint64_t s1_bytes, uint64_t s2_bytes, uint32_t b0, uint32_t b1, uint32_t b2)
{
    const uint64_t dims[3] = {d0, d1, d2};
    const uint64_t strides[2] = {s1_bytes, s2_bytes};
    const uint32_t box[3] = {b0, b1, b2};
    return encode_tmap(tm, base, 3, dims, strides, box);
}

template <int CLN, int BNT, bool DEEP, bool STG2, bool COMPACT>
caat_status launch_fwd_v(const CUtensorMap &tmX, const CUtensorMap &tmW, const YMaps &ym, const FwdParams &p,
                         cudaStream_t s)
{
    constexpr bool PAIR = CLN > 1;
    auto kern = rowpar_fwd_tc_kernel<CLN, BNT, DEEP, STG2, COMPACT>;
    static_assert(smem_bytes<CLN, BNT, DEEP, STG2>() + bitmap_bytes(192) <= 227 * 1024,
                  "shared memory beyond the per-CTA limit");
    const size_t smem = smem_bytes<CLN, BNT, DEEP, STG2>() + bitmap_bytes(p.h);
    if (smem > 227 * 1024) return CAAT_ERR_UNSUPPORTED;
    if (prepare_kernel_smem((const void *)kern, (int)smem) != CAAT_OK) return CAAT_ERR_CUDA;
    const int per = CLN;
    const int num_mg = (p.num_m + CLN - 1) / CLN;
    // work items available: whole tiles, plus t pieces per NO_S tile when balanced
    const int num_units = p.balanced ? num_mg * p.n_whole + num_mg * (p.num_n - p.n_whole) * p.t
                                     : num_mg * p.num_n;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = per;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(NUM_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int groups = num_sms() / per;
    if (PAIR) {
        cfg.gridDim = dim3(groups * per);
        const int active = max_active_clusters((const void *)kern, cfg);
        if (active < 1) return CAAT_ERR_UNSUPPORTED;
        if (active < groups) groups = active;
    }
    if (groups > num_units) groups = num_units;
    cfg.gridDim = dim3(groups * per);
    // a programmatic dependent of the previous launch in the stream (CAAT_PDL=0: a
    // plain launch); the kernel waits for that grid before touching memory
    cudaLaunchAttribute attr2[2] = {attr[0], {}};
    const char *pdl_env = std::getenv("CAAT_PDL");
    if (pdl_env == nullptr || std::strcmp(pdl_env, "0") != 0) {
        attr2[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr2[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr2;
        cfg.numAttrs = 2;
    }
    if (cudaLaunchKernelEx(&cfg, kern, tmX, tmW, ym, p) != cudaSuccess) return CAAT_ERR_CUDA;
    note_launch("rowpar_fwd_tc");
    return cudaGetLastError() == cudaSuccess ? CAAT_OK : CAAT_ERR_CUDA;
}

template <int CLN, int BNT, bool DEEP = false, bool STG2 = false>
caat_status launch_fwd(const CUtensorMap &tmX, const CUtensorMap &tmW, const YMaps &ym, const FwdParams &p,
                       cudaStream_t s, bool compact)
{
    return compact ? launch_fwd_v<CLN, BNT, DEEP, STG2, true>(tmX, tmW, ym, p, s)
                   : launch_fwd_v<CLN, BNT, DEEP, STG2, false>(tmX, tmW, ym, p, s);
}

}  // namespace

caat_status launch_rowpar_fwd_tc(int t, int64_t N, int64_t K, int64_t h, const void *X, int64_t ldx,
                                 const void *W, int64_t ldw, const MutPtrs &Y, int64_t ldy,
                                 const int32_t *sel, int64_t n_sel, cudaStream_t s, void *YS, int64_t ldys)
{
    const int64_t kt = K / t;
    const bool compact = YS != nullptr;
    // shapes and alignments this kernel takes; anything else goes to another kernel
    if (kt < BK || kt % 8 != 0 || ldx % 8 != 0 || ldw % 8 != 0 || ldy % 8 != 0) return CAAT_ERR_UNSUPPORTED;
    if (compact && (sel != nullptr || n_sel % 64 != 0 || ldys % 8 != 0 || (uintptr_t)YS % 16 != 0))
        return CAAT_ERR_UNSUPPORTED;
    // (h < 256 only as 192-wide single-CTA tiles)
    if (h % 8 != 0 || h < (h % 192 == 0 ? 192 : BN) || h > MAX_H_TC || N < 16 || N > (int64_t)INT32_MAX)
        return CAAT_ERR_UNSUPPORTED;
    if (t > MAX_T_TC) return CAAT_ERR_UNSUPPORTED;
    if ((uintptr_t)X % 16 != 0 || (uintptr_t)W % 16 != 0) return CAAT_ERR_UNSUPPORTED;
    for (int r = 0; r < t; ++r)
        if ((uintptr_t)Y.p[r] % 16 != 0) return CAAT_ERR_UNSUPPORTED;
    YMaps ym;
    const int64_t h_out = compact ? h - n_sel : h;     // channels of each rank's own output
    for (int r = 0; r < t; ++r) {
        if (h_out == 0) { ym.m[r] = CUtensorMap{}; continue; }   // (never stored to)
        const uint64_t dims[2] = {(uint64_t)h_out, (uint64_t)N};
        const uint64_t str[1] = {(uint64_t)ldy * 2};
        const uint32_t box[2] = {64, 32};
        if (!encode_tmap(&ym.m[r], Y.p[r], 2, dims, str, box)) return CAAT_ERR_UNSUPPORTED;
    }
    ym.s = CUtensorMap{};
    if (compact && n_sel > 0) {
        const uint64_t dims[2] = {(uint64_t)n_sel, (uint64_t)N};
        const uint64_t str[1] = {(uint64_t)ldys * 2};
        const uint32_t box[2] = {64, 32};
        if (!encode_tmap(&ym.s, YS, 2, dims, str, box)) return CAAT_ERR_UNSUPPORTED;
    }
    // CTAs per cluster: a CTA pair when there are at least two 128-row blocks,
    // else one CTA per tile.  Short shards (k_t <= 384) make the t output copies
    // the bottleneck; there the finer single-CTA tiles balance the writes better
    // over the SMs.  (override: CAAT_FWD_CLUSTER=1|2)
    const int64_t nm = (N + BM - 1) / BM;
    int cln = kt <= 384 ? 1 : (nm >= 2 ? 2 : 1);
    if (const char *e = std::getenv("CAAT_FWD_CLUSTER")) {
        const int v = std::atoi(e);
        if ((v == 1 || v == 2) && v <= nm) cln = v;
    }

    CUtensorMap tmX;
    if (!encode_3d(&tmX, X, (uint64_t)kt, (uint64_t)t, (uint64_t)N, (uint64_t)kt * 2, (uint64_t)ldx * 2,
                   BK, 1, BM))
        return CAAT_ERR_UNSUPPORTED;

    FwdParams p{};
    p.Y = Y;
    p.ldy = ldy;
    p.N = N;
    p.h = h;
    p.t = t;
    p.nkb = (int)((kt + BK - 1) / BK);
    p.num_m = (int)((N + BM - 1) / BM);
    // Work-unit order: row-block-major when X is large and has many more rows than
    // W has channels, and a contiguous S ends on a tile edge -- the channel blocks
    // of a row block then run in the same round and read X from DRAM once (1.1B:
    // -4 to -6 %, 130M down-proj: -2 %); channel-block-major otherwise, which keeps
    // W tiles hot when N ~ h (7B prefill) or X fits in L2 anyway.
    // (override: CAAT_FWD_ORDER=m|n)
    // (decided per tile width below: only without MIXED tiles, whose slow per-shard
    // epilogues would then pile up on the CTAs that run two units)
    const bool mmajor_size = N * K * 2 >= ((int64_t)32 << 20) && N >= 2 * h;
    const char *order_env = std::getenv("CAAT_FWD_ORDER");
    const char *sched_env = std::getenv("CAAT_FWD_SCHED");
    p.sel = sel;
    p.n_sel = n_sel;
    p.wait_ns = g_wait_ns.load();
    p.inject = g_inject.load();
    // Tile width of the single-CTA mode: 192 channels instead of 256 when h is a
    // multiple of 192, the tiles then take fewer SM-rounds of work (rounds x
    // width), and a contiguous S ends on a tile edge (no MIXED tiles).  At the
    // 130M shapes (h = 768, S = [0, 384)) this is 256 tiles of 3/4 the work in
    // the same two rounds as 192 full tiles.  (override: CAAT_FWD_BN=192|256)
    auto rounds = [&](int64_t bn) { return (p.num_m * ((h + bn - 1) / bn) + num_sms() - 1) / num_sms(); };
    bool bn192 = h % 192 == 0 && rounds(192) * 192 < rounds(256) * 256 && (sel != nullptr || n_sel % 192 == 0);
    if (const char *e = std::getenv("CAAT_FWD_BN")) {
        const int v = std::atoi(e);
        if (v == 192 && h % 192 == 0) bn192 = true;
        if (v == 256 && h >= BN) bn192 = false;
    }
    if (h < BN) bn192 = true;
    const char *bn_env = std::getenv("CAAT_FWD_BN");
    const bool bn192_clusters = bn_env != nullptr && std::atoi(bn_env) == 192 && h % 192 == 0;
    for (;; cln >>= 1) {
        if (cln > 1 && h < BN) continue;           // the cluster modes need 256 channels
        const int bn = ((cln == 1 && bn192) || (cln > 1 && bn192_clusters)) ? 192 : BN;
        p.mmajor = (mmajor_size && sel == nullptr && n_sel % bn == 0) ? 1 : 0;
        if (order_env != nullptr) p.mmajor = order_env[0] == 'm' ? 1 : 0;
        p.num_n = (int)((h + bn - 1) / bn);
        // Balanced schedule where the host knows every tile's class: a contiguous S
        // (passed by its size) with t > 1 and at least one channel block outside
        // S.  A block is NO_S when it starts at or after s, whole otherwise (FULL_S
        // when it ends by s, MIXED across the boundary).  The pieces run in equal
        // runs around each worker's whole tiles.  (override: CAAT_FWD_SCHED=rounds
        // keeps every tile whole; CAAT_FWD_SCHED=first runs the whole tiles first)
        p.balanced = 0;
        p.n_whole = p.num_n;
        // A whole tile of S costs about t pieces when it writes t copies.  With the
        // compact outputs it writes one, so it is worth fewer pieces the shorter
        // the shards: measured best near k-blocks / 2 + 2 (130M out-proj 35.3 ->
        // 29.2 us, 1.1B 72.4 -> 66.0, 7B 104.1 -> 98.4; t for the long shards of
        // the down-projections).
        p.wgt = compact ? (p.nkb / 2 + 2 < t ? p.nkb / 2 + 2 : t) : t;
        if (const char *e = std::getenv("CAAT_FWD_WGT")) {
            const int v = std::atoi(e);
            if (v >= 1 && v <= t) p.wgt = v;
        }
        const bool rounds_env = sched_env != nullptr && sched_env[0] == 'r';
        // An index list of S with 0 < |S| < h (a random S): its tiles would be MIXED
        // -- per-shard epilogues, the S channels summed in TMEM across shards, and
        // masked stores of the sums to every rank -- and MIXED tiles cannot be cut
        // into pieces.  Instead every tile runs as per-shard pieces (each rank's
        // partial, all channels) and the S channels are then summed over the ranks
        // in place by the standalone partial reduce (rank-order fp32 fold of the
        // bf16 partials).  (CAAT_FWD_SCHED=rounds keeps the MIXED tiles)
        const bool pieces_then_reduce = sel != nullptr && n_sel > 0 && n_sel < h && t > 1 &&
                                        p.num_n <= MAX_NB && !rounds_env;
        if (pieces_then_reduce) {
            for (int nb = 0; nb < p.num_n; ++nb) p.nbl[nb] = (uint8_t)nb;
            p.n_whole = 0;
            p.balanced = 2;
        }
        if (sel == nullptr && t > 1 && p.num_n <= MAX_NB && !rounds_env) {
            int nw = 0, ns = 0;
            uint8_t no_s[MAX_NB];
            for (int nb = 0; nb < p.num_n; ++nb) {
                if ((int64_t)nb * bn >= n_sel) no_s[ns++] = (uint8_t)nb;
                else p.nbl[nw++] = (uint8_t)nb;
            }
            if (ns > 0) {
                for (int k = 0; k < ns; ++k) p.nbl[nw + k] = no_s[k];
                p.n_whole = nw;
                p.balanced = (sched_env != nullptr && sched_env[0] == 'f') ? 1 : 2;
            }
        }
        if ((int64_t)p.num_m * p.num_n > INT32_MAX / 4) return CAAT_ERR_UNSUPPORTED;
        CUtensorMap tmW;
        const uint32_t wrows = cln == 1 ? bn : bn / 2;
        if (!encode_3d(&tmW, W, (uint64_t)kt, (uint64_t)t, (uint64_t)h, (uint64_t)kt * 2, (uint64_t)ldw * 2,
                       BK, 1, wrows))
            return CAAT_ERR_UNSUPPORTED;
        caat_status st;
        if (bn == 192) {
            // the deeper ring (5 stages, one staging buffer per warp) for shards of
            // 4 or more k-blocks (override: CAAT_FWD_DEEP=0|1)
            bool deep = p.nkb >= 4;
            if (const char *e = std::getenv("CAAT_FWD_DEEP")) deep = e[0] == '1';
            st = cln == 2 ? launch_fwd<2, 192>(tmX, tmW, ym, p, s, compact)
               : (deep ? launch_fwd<1, 192, true>(tmX, tmW, ym, p, s, compact)
                       : launch_fwd<1, 192>(tmX, tmW, ym, p, s, compact));
        }
        else {
            // two staging buffers where the bitmap leaves room (CAAT_FWD_STG=1: one)
            const char *stg_env = std::getenv("CAAT_FWD_STG");
            const bool one = stg_env != nullptr && stg_env[0] == '1';
            if (cln == 2) {
                const bool stg2 = !one && smem_bytes<2, BN, false, true>() + bitmap_bytes(h) <= 227 * 1024;
                st = stg2 ? launch_fwd<2, BN, false, true>(tmX, tmW, ym, p, s, compact)
                          : launch_fwd<2, BN>(tmX, tmW, ym, p, s, compact);
            } else {
                const bool stg2 = !one && smem_bytes<1, BN, false, true>() + bitmap_bytes(h) <= 227 * 1024;
                st = stg2 ? launch_fwd<1, BN, false, true>(tmX, tmW, ym, p, s, compact)
                          : launch_fwd<1, BN>(tmX, tmW, ym, p, s, compact);
            }
        }
        if (st == CAAT_OK && pieces_then_reduce) {
            ConstPtrs yin{};
            for (int r = 0; r < t; ++r) yin.p[r] = Y.p[r];
            st = launch_pcr(t, N, h, CAAT_BF16, yin, ldy, Y, ldy, true, sel, n_sel, s);
            if (st == CAAT_OK) note_launch("rowpar_fwd_tc", 0);   // the call's main kernel
            return st;
        }
        // a cluster shape that cannot be co-resident falls back to a smaller one
        if (st != CAAT_ERR_UNSUPPORTED || cln == 1) return st;
    }
}

}  // namespace caat

extern "C" caat_status caat_debug_set_wait(uint64_t limit_ns, caat_inject inject)
{
    if (limit_ns != 0 && (limit_ns < 1000ull || limit_ns > 10000000000ull)) return CAAT_ERR_INVALID_ARG;
    if (inject != CAAT_INJECT_NONE && inject != CAAT_INJECT_SKIP_LOADS) return CAAT_ERR_INVALID_ARG;
    caat::g_wait_ns.store(limit_ns == 0 ? caat::WAIT_LIMIT_NS : limit_ns);
    caat::g_inject.store((int)inject);
    return CAAT_OK;
}
