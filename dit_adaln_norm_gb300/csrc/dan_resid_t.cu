// dan_resid_t.cu -- residual gating with the residual stream in the
// [B, hidden, tokens] layout.
//
// "SGLang diffusion fused-op package guide", norm variants, residual
// gating: the transposed dense path reads the update through shared-memory
// tiles in its logical row-major order and keeps the residual reads and the
// output writes coalesced on their [B, hidden, tokens] layout (no
// .contiguous() copy of the residual).  Per element
//   r_out[b, d, t] = bf16(rn(r[b, d, t] + bf16(rn(gate[b, d] * h[b, t, d])))).
//
// T % 8 == 0 (every residual row 16-byte aligned): a persistent kernel,
// six CTAs of 64 threads per SM, each taking a contiguous run of
// 64-channel x 64-token tiles (tokens fastest, so a CTA streams along its
// 64 residual rows; measured faster than interleaving the CTAs' tiles, or
// than running channels fastest).  Both inputs of a tile are staged in
// shared memory by 16-byte asynchronous copies, one tile ahead: the update
// as 64 token rows of 128 bytes, its 16-byte chunks XOR-swizzled by the
// row's token octet, the residual as 64 channel rows of 128 bytes.  Each
// thread then takes one channel octet x one token octet: eight 16-byte
// shared loads of the update (one per token; the swizzle puts the eight
// lanes of a load phase on eight different bank groups), eight of the
// residual (one per channel), and eight 16-byte stores of r_out, each
// eight lanes covering 128 contiguous bytes of one residual row.  The
// product bf16(gate * h) is formed on channel pairs, as the update holds
// them, and regrouped into token pairs with byte permutes before the add.
//
// Other T (residual rows not 16-byte aligned): one 64 x 64 tile per CTA,
// token pairs on 4-byte boundaries with the lanes of a warp on consecutive
// pairs, the residual words loaded together with the update tile.
#include "dan_device.cuh"
#include "dan_internal.h"
#include "dan_ring.cuh"

namespace dan {

namespace {

constexpr int kTile = 64;          // channels and tokens per tile
constexpr int kResidThreads = 128; // four warps per 64 x 64 tile
constexpr int kResidCtas = 8;      // resident CTAs per SM the register budget allows

struct ResidParams {
    const uint16_t *r;
    const uint4 *h;
    const uint16_t *gate;
    uint16_t *r_out;
    int64_t T, D, vs;
    unsigned tiles_t, tiles_d, tiles; // tile counts (checked on the host to fit 32 bits)
};

// (a, b) -> the 16-bit halves: low of both, high of both.
__device__ __forceinline__ uint32_t lows(uint32_t a, uint32_t b) { return __byte_perm(a, b, 0x5410); }
__device__ __forceinline__ uint32_t highs(uint32_t a, uint32_t b) { return __byte_perm(a, b, 0x7632); }

struct TileAt {
    unsigned b, d0, t0;
};

// Tile i of the (batch, channel tile, token tile) order, tokens fastest,
// for tiles of kTile tokens.
__device__ __forceinline__ TileAt tile_at(const ResidParams &p, unsigned i)
{
    const unsigned tt = i % p.tiles_t, rest = i / p.tiles_t;
    const unsigned dt = rest % p.tiles_d, b = rest / p.tiles_d;
    return TileAt{b, dt * kTile, tt * kTile};
}

// Any T: one 64 x 64 tile per CTA of 128 threads (tokens fastest in
// the grid), up to kResidCtas CTAs per SM.  The update tile sits
// in shared memory at a pitch of 33 words; each warp walks channel rows,
// lane k on the k-th 4-byte-aligned token pair of the row's segment (so a
// warp's residual loads and stores cover 128 contiguous bytes), with single
// elements, as 2-byte accesses, where a segment starts or ends off a pair.
__global__ void __launch_bounds__(kResidThreads, kResidCtas) gated_residual_t_kernel(const ResidParams p)
{
    constexpr int kPitchW = kTile / 2 + 1; // words per update row: 32 channel pairs + 1
    __shared__ uint32_t s_h[kTile * kPitchW]; // update tile: [token][channel pair]
    __shared__ uint32_t s_g[kTile];           // gate of each channel (low half)

    grid_dependency_wait(); // no global access above this line
    allow_dependents();
    const int64_t T = p.T, D = p.D;
    const int tid = threadIdx.x;
    const TileAt at = tile_at(p, blockIdx.x);

    // Update tile: 64 rows x 8 chunks of 16 bytes; chunks outside the
    // tensor read as zero (their products are never stored).
    {
        const int ch = tid & 7;
        const bool col_in = (int64_t)at.d0 + 8 * ch < D; // D % 8 == 0: whole chunk
        const uint4 *h = p.h + (((int64_t)at.b * T + at.t0) * D + at.d0) / 8 + ch;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int row = (tid >> 3) + 16 * j;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (col_in && (int64_t)at.t0 + row < T) v = ld_stream(h + (int64_t)row * (D / 8));
            uint32_t *dst = s_h + row * kPitchW + 4 * ch;
            dst[0] = v.x;
            dst[1] = v.y;
            dst[2] = v.z;
            dst[3] = v.w;
        }
    }
    if (tid < kTile) {
        const int64_t d = (int64_t)at.d0 + tid;
        s_g[tid] = d < D ? (uint32_t)p.gate[(int64_t)at.b * p.vs + d] : 0u;
    }

    // Token pairs on 4-byte boundaries: (2k, 2k+1) when a row segment starts
    // on one, else (2k+1, 2k+2) and token 0 alone.  The residual words are
    // loaded before the barrier, so they are in flight with the update tile.
    const int warp = tid >> 5, lane = tid & 31;
    const int nt = (int)(T - at.t0 < kTile ? T - at.t0 : kTile); // tokens of the tile
    constexpr int kRows = kTile / 4;                               // channel rows per warp
    uint32_t rw[kRows], r0[kRows];
#pragma unroll
    for (int j = 0; j < kRows; ++j) {
        const int dl = warp + 4 * j;
        rw[j] = r0[j] = 0u;
        if ((int64_t)at.d0 + dl >= D) continue;
        const int64_t rb = ((int64_t)at.b * D + at.d0 + dl) * T + at.t0; // r[b][d][t0]
        const int odd = (int)(rb & 1), t = 2 * lane + odd;
        if (t + 1 < nt) rw[j] = *reinterpret_cast<const uint32_t *>(p.r + rb + t);
        else if (t < nt) rw[j] = p.r[rb + t];
        if (odd && lane == 0) r0[j] = p.r[rb];
    }
    __syncthreads();

    // update element of token tl, channel dl (low half)
    auto hval = [&](int tl, int dl) -> uint32_t {
        const uint32_t hw = s_h[tl * kPitchW + (dl >> 1)];
        return (dl & 1) ? hw >> 16 : hw & 0xFFFFu;
    };
#pragma unroll
    for (int j = 0; j < kRows; ++j) {
        const int dl = warp + 4 * j; // channel within the tile
        if ((int64_t)at.d0 + dl >= D) break; // warp-uniform
        const uint32_t g = s_g[dl], g2 = g | (g << 16);
        const int64_t rb = ((int64_t)at.b * D + at.d0 + dl) * T + at.t0;
        const int odd = (int)(rb & 1), t = 2 * lane + odd;
        if (t + 1 < nt) {
            const uint32_t h2 = hval(t, dl) | (hval(t + 1, dl) << 16);
            *reinterpret_cast<uint32_t *>(p.r_out + rb + t) = gated_word(rw[j], g2, h2);
        } else if (t < nt) {
            p.r_out[rb + t] = (uint16_t)gated_word(rw[j], g, hval(t, dl));
        }
        if (odd && lane == 0) p.r_out[rb] = (uint16_t)gated_word(r0[j], g, hval(0, dl));
    }
}

// ------------------------------------------------ the pipelined kernel

constexpr int kPD = 64;         // channels per tile
constexpr int kPT = 64;        // tokens per tile
constexpr int kRC = kPT / 8;    // token octets per tile (16-byte chunks per residual row)
constexpr int kHC = kPD / 8;    // channel octets per tile (16-byte chunks per update row)
constexpr int kPThreads = kHC * kRC; // one thread per channel octet x token octet
constexpr int kPipeCtas = 6;    // CTAs per SM (shared memory allows six)
constexpr int kStages = 2;      // tiles in shared memory (kStages - 1 in flight)
constexpr int kStageH = kPT * kPD / 8;  // 16-byte chunks of the update per tile
constexpr int kStageR = kPD * kPT / 8;  // 16-byte chunks of the residual per tile

struct PipeTile {
    unsigned b, d0, t0;
};

// Tile i of the (batch, channel tile, token tile) order, tokens fastest.
__device__ __forceinline__ PipeTile pipe_tile(const ResidParams &p, unsigned i)
{
    const unsigned tt = i % p.tiles_t, rest = i / p.tiles_t;
    const unsigned dt = rest % p.tiles_d, b = rest / p.tiles_d;
    return PipeTile{b, dt * kPD, tt * kPT};
}

// Issue this thread's asynchronous copies of tile i into stage buffers
// (sh, sr).  Chunks outside the tensor are not copied: the outputs that
// would read them are never stored.
__device__ __forceinline__ void pipe_issue(const ResidParams &p, unsigned i, uint4 *sh, uint4 *sr)
{
    const PipeTile at = pipe_tile(p, i);
    const int tid = threadIdx.x;
    const int64_t T = p.T, D = p.D;
    {   // update: kPT token rows x kHC chunks; chunk c of row k goes to slot c ^ ((k >> 3) & 7)
        const int c = tid % kHC;
        if ((int64_t)at.d0 + 8 * c < D) {
            const uint4 *src = p.h + (((int64_t)at.b * T + at.t0) * D + at.d0) / 8 + c;
#pragma unroll
            for (int j = 0; j < kStageH / kPThreads; ++j) {
                const int k = tid / kHC + (kPThreads / kHC) * j;
                if ((int64_t)at.t0 + k < T)
                    cp_async16(sh + k * kHC + (c ^ ((k >> 3) & 7)), src + (int64_t)k * (D / 8));
            }
        }
    }
    {   // residual: 64 channel rows x kRC chunks
        const int u = tid % kRC;
        if ((int64_t)at.t0 + 8 * u < T) {
            const uint16_t *src = p.r + ((int64_t)at.b * D + at.d0) * T + at.t0 + 8 * u;
#pragma unroll
            for (int j = 0; j < kStageR / kPThreads; ++j) {
                const int k = tid / kRC + (kPThreads / kRC) * j;
                if ((int64_t)at.d0 + k < D) cp_async16(sr + k * kRC + u, src + (int64_t)k * T);
            }
        }
    }
}

// CTA c takes tiles [c*N/G, (c+1)*N/G).  Requires T % 8 == 0.
__global__ void __launch_bounds__(kPThreads, kPipeCtas) gated_residual_t_pipe_kernel(const ResidParams p)
{
    extern __shared__ __align__(128) uint4 s_pipe[]; // kStages x (update, residual)
    grid_dependency_wait(); // no global access above this line
    allow_dependents();
    const unsigned G = gridDim.x;
    const unsigned first = (unsigned)((uint64_t)blockIdx.x * p.tiles / G);
    const unsigned n = (unsigned)((uint64_t)(blockIdx.x + 1) * p.tiles / G) - first;
    auto tile_of = [&](unsigned i) { return first + i; };
    auto stage_h = [&](unsigned i) { return s_pipe + (i % kStages) * (kStageH + kStageR); };
    auto stage_r = [&](unsigned i) { return stage_h(i) + kStageH; };
#pragma unroll
    for (int s = 0; s < kStages - 1; ++s) {
        if ((unsigned)s < n) pipe_issue(p, tile_of(s), stage_h(s), stage_r(s));
        cp_async_commit(); // one group per tile, empty past the end
    }
    const int o = threadIdx.x / kRC; // channel octet of the tile
    const int v = threadIdx.x % kRC; // token octet of the tile
    const int64_t T = p.T, D = p.D;
    for (unsigned i = 0; i < n; ++i) {
        cp_async_wait<kStages - 2>(); // this thread's copies of tile i have landed
        __syncthreads();              // everyone's have; everyone is done with tile i - 1
        if (i + kStages - 1 < n)
            pipe_issue(p, tile_of(i + kStages - 1), stage_h(i + kStages - 1), stage_r(i + kStages - 1));
        cp_async_commit();

        const PipeTile at = pipe_tile(p, tile_of(i));
        const int64_t d = (int64_t)at.d0 + 8 * o, t = (int64_t)at.t0 + 8 * v;
        if (d >= D || t >= T) continue; // D, T multiples of 8: whole octets in or out
        const uint4 g = *reinterpret_cast<const uint4 *>(p.gate + (int64_t)at.b * p.vs + d);
        const uint4 *sh = stage_h(i), *sr = stage_r(i);
        // gh[k]: channel pairs of token t + k, bf16(gate * h)
        uint4 gh[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const uint4 hv = sh[(8 * v + k) * kHC + (o ^ (v & 7))];
            gh[k] = make_uint4(hmul2(g.x, hv.x), hmul2(g.y, hv.y), hmul2(g.z, hv.z), hmul2(g.w, hv.w));
        }
        uint16_t *out = p.r_out + ((int64_t)at.b * D + d) * T + t;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const uint4 rv = sr[(8 * o + c) * kRC + v];
            // channel c, token pair (2q, 2q+1): low (c even) or high halves
            // of channel pair c / 2 in the two tokens' products
            auto pair = [&](int q) -> uint32_t {
                const uint32_t a = word(gh[2 * q], c >> 1), b = word(gh[2 * q + 1], c >> 1);
                return (c & 1) ? highs(a, b) : lows(a, b);
            };
            const uint4 res = make_uint4(hadd2(rv.x, pair(0)), hadd2(rv.y, pair(1)),
                                         hadd2(rv.z, pair(2)), hadd2(rv.w, pair(3)));
            st_stream(reinterpret_cast<uint4 *>(out + (int64_t)c * T), res);
        }
    }
    cp_async_wait_all(); // no copy outlives the CTA
}

} // namespace

cudaError_t launch_gated_residual_transposed(const ResidProblem &q, cudaStream_t s)
{
    ResidParams p;
    p.r = static_cast<const uint16_t *>(q.r);
    p.h = static_cast<const uint4 *>(q.h);
    p.gate = static_cast<const uint16_t *>(q.gate);
    p.r_out = static_cast<uint16_t *>(q.r_out);
    p.T = q.T;
    p.D = q.D;
    p.vs = q.vs;
    const int64_t tt = (q.T + kTile - 1) / kTile, td = (q.D + kTile - 1) / kTile;
    if (q.B * tt * td >= (int64_t(1) << 31)) return cudaErrorInvalidValue; // beyond 32-bit tile ids
    p.tiles_t = (unsigned)tt;
    p.tiles_d = (unsigned)td;
    p.tiles = (unsigned)(q.B * tt * td);
    if (q.T % 8 == 0) {
        const int64_t ptiles = q.B * ((q.D + kPD - 1) / kPD) * ((q.T + kPT - 1) / kPT);
        p.tiles_t = (unsigned)((q.T + kPT - 1) / kPT);
        p.tiles_d = (unsigned)((q.D + kPD - 1) / kPD);
        p.tiles = (unsigned)ptiles; // at most the 64 x 64 tile count checked above
        constexpr int smem = kStages * (kStageH + kStageR) * 16;
        const cudaError_t e = allow_dynamic_smem(reinterpret_cast<const void *>(gated_residual_t_pipe_kernel), smem);
        if (e != cudaSuccess) return e;
        const int64_t cap = (int64_t)sm_count() * kPipeCtas;
        const int grid = (int)(ptiles < cap ? ptiles : cap);
        return launch_overlapped(gated_residual_t_pipe_kernel, grid, kPThreads, smem, s, p);
    }
    return launch_overlapped(gated_residual_t_kernel, (int)p.tiles, kResidThreads, 0, s, p);
}

} // namespace dan
