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
// 64-token x 64-channel tiles: the update tile (64 token rows of 128
// contiguous bytes) is read with 16-byte loads into shared memory with a
// padded row pitch of 33 words, so that a warp reading one channel pair
// across 32 tokens touches 32 different banks; each warp takes channel
// pairs, each lane two neighbouring tokens of both channels (4-byte loads
// and stores of the residual, 128 contiguous bytes per warp).  A CTA's
// next tile is loaded into registers while the current one is computed.
#include "dan_device.cuh"
#include "dan_internal.h"
#include "dan_ring.cuh"

namespace dan {

namespace {

constexpr int kTile = 64;   // tokens and channels per tile
constexpr int kPitchW = 33; // shared-memory words per update row (32 of data)
constexpr int kResidThreads = 256;

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

// Per-thread offsets that do not change from tile to tile.
struct ResidLane {
    int64_t hoff[2]; // update chunk j: token row (c >> 3) * D/8 + chunk (c & 7), in uint4
    int64_t roff[4]; // channel pair j: (2 * (warp + 8 j)) * T + 2 * lane, in elements
    int ht[2], hc[2]; // update chunk j: token row and chunk within the tile
};

// Registers of one tile in flight: its coordinates and this thread's update
// chunks and, for a full tile with even T, its residual words.
struct ResidTile {
    uint4 h[2];
    uint32_t r0[4], r1[4];
    int64_t b, d0, t0;
    int64_t rbase; // element index of r[b][d0][t0]
    bool full;     // the whole 64 x 64 tile lies inside the tensor
};

// Tile order: within a batch, bands of kBand token tiles; in a band, the
// channel tiles, and in each channel tile the band's token tiles, so the
// tiles in flight at once cover whole update rows and runs of each
// residual row.  32-bit tile arithmetic.
constexpr unsigned kBand = 16;

__device__ __forceinline__ void tile_coords(const ResidParams &p, unsigned tile, ResidTile &u)
{
    const unsigned per_b = p.tiles_d * p.tiles_t;
    const unsigned b = tile / per_b, rem = tile - b * per_b;
    const unsigned full = p.tiles_t / kBand, in_full = full * kBand * p.tiles_d;
    unsigned dt, tt;
    if (rem < in_full) {
        const unsigned band = rem / (kBand * p.tiles_d), r2 = rem - band * (kBand * p.tiles_d);
        dt = r2 / kBand;
        tt = band * kBand + (r2 - dt * kBand);
    } else { // the last, narrower band
        const unsigned w = p.tiles_t - full * kBand, r2 = rem - in_full;
        dt = r2 / w;
        tt = full * kBand + (r2 - dt * w);
    }
    u.b = b;
    u.d0 = (int64_t)dt * kTile;
    u.t0 = (int64_t)tt * kTile;
    u.rbase = (p.D * u.b + u.d0) * p.T + u.t0;
    u.full = u.t0 + kTile <= p.T && u.d0 + kTile <= p.D;
}

// Issue the loads of a tile: the update chunks always (D % 8 == 0, so a
// chunk is wholly inside or outside its row), the residual words for a
// full tile when T is even (rows 4-byte aligned).
template <bool EVEN_T>
__device__ __forceinline__ void tile_load(const ResidParams &p, const ResidLane &L, unsigned tile,
                                          ResidTile &u)
{
    tile_coords(p, tile, u);
    const uint4 *h = p.h + ((p.T * u.b + u.t0) * p.D + u.d0) / 8;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        if (u.full || (u.t0 + L.ht[j] < p.T && u.d0 + 8 * L.hc[j] < p.D))
            u.h[j] = ld_stream(h + L.hoff[j]);
        else
            u.h[j] = make_uint4(0, 0, 0, 0);
    }
    if (EVEN_T && u.full) {
        const uint16_t *r = p.r + u.rbase;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            u.r0[j] = *reinterpret_cast<const uint32_t *>(r + L.roff[j]);
            u.r1[j] = *reinterpret_cast<const uint32_t *>(r + L.roff[j] + p.T);
        }
    }
}

// The gated residual of one tile (its update chunks, and residual words
// when loaded, in u).
template <bool EVEN_T>
__device__ __forceinline__ void tile_compute(const ResidParams &p, const ResidLane &L,
                                             const ResidTile &u, uint32_t *s_h, uint32_t *s_g,
                                             int warp, int lane)
{
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        uint32_t *dst = s_h + L.ht[j] * kPitchW + 4 * L.hc[j];
        dst[0] = u.h[j].x;
        dst[1] = u.h[j].y;
        dst[2] = u.h[j].z;
        dst[3] = u.h[j].w;
    }
    if (threadIdx.x < kTile / 2) {
        const int64_t d = u.d0 + 2 * threadIdx.x;
        s_g[threadIdx.x] =
            d < p.D ? *reinterpret_cast<const uint32_t *>(p.gate + u.b * p.vs + d) : 0u;
    }
    __syncthreads();

    const int t = 2 * lane; // this lane's tokens t0 + t, t0 + t + 1
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int pr = warp + 8 * j;
        const uint32_t g2 = s_g[pr];
        const uint32_t gd = __byte_perm(g2, 0, 0x1010), gd1 = __byte_perm(g2, 0, 0x3232);
        const uint32_t ht = s_h[t * kPitchW + pr], ht1 = s_h[(t + 1) * kPitchW + pr];
        const uint32_t hd = lows(ht, ht1), hd1 = highs(ht, ht1); // (tokens t, t+1) per channel
        uint16_t *out = p.r_out + u.rbase + L.roff[j];
        if (EVEN_T && u.full) {
            *reinterpret_cast<uint32_t *>(out) = gated_word(u.r0[j], gd, hd);
            *reinterpret_cast<uint32_t *>(out + p.T) = gated_word(u.r1[j], gd1, hd1);
        } else if (u.d0 + 2 * pr < p.D && u.t0 + t < p.T) {
            // an edge tile, or rows not 4-byte aligned: token by token
            const uint16_t *in = p.r + u.rbase + L.roff[j];
            const bool two = u.t0 + t + 1 < p.T;
            const uint32_t r0 = in[0] | (two ? (uint32_t)in[1] << 16 : 0u);
            const uint32_t r1 = in[p.T] | (two ? (uint32_t)in[p.T + 1] << 16 : 0u);
            const uint32_t w0 = gated_word(r0, gd, hd), w1 = gated_word(r1, gd1, hd1);
            out[0] = (uint16_t)w0;
            out[p.T] = (uint16_t)w1;
            if (two) {
                out[1] = (uint16_t)(w0 >> 16);
                out[p.T + 1] = (uint16_t)(w1 >> 16);
            }
        }
    }
    __syncthreads(); // the tile's shared memory is reused by the next tile
}

// EVEN_T: T is even, so every residual row starts 4-byte aligned and a
// lane's token pair can move as one word.  Each CTA walks its tiles two at
// a time, the next tile's loads issued before the current one is computed.
template <bool EVEN_T>
__global__ void __launch_bounds__(kResidThreads, 4) gated_residual_t_kernel(const ResidParams p)
{
    __shared__ uint32_t s_h[kTile * kPitchW]; // update tile: [token][channel pair]
    __shared__ uint32_t s_g[kTile / 2];       // gate pairs

    grid_dependency_wait(); // no global access above this line
    allow_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    ResidLane L;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const int c = threadIdx.x + kResidThreads * j;
        L.ht[j] = c >> 3;
        L.hc[j] = c & 7;
        L.hoff[j] = (int64_t)L.ht[j] * (p.D / 8) + L.hc[j];
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) L.roff[j] = (int64_t)(2 * (warp + 8 * j)) * p.T + 2 * lane;

    unsigned tile = blockIdx.x;
    if (tile >= p.tiles) return;
    ResidTile A, Bt;
    tile_load<EVEN_T>(p, L, tile, A);
    for (;;) {
        const unsigned t1 = tile + gridDim.x, t2 = t1 + gridDim.x;
        if (t1 < p.tiles) tile_load<EVEN_T>(p, L, t1, Bt);
        tile_compute<EVEN_T>(p, L, A, s_h, s_g, warp, lane);
        if (t1 >= p.tiles) break;
        if (t2 < p.tiles) tile_load<EVEN_T>(p, L, t2, A);
        tile_compute<EVEN_T>(p, L, Bt, s_h, s_g, warp, lane);
        if (t2 >= p.tiles) break;
        tile = t2;
    }
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
    const unsigned cap = (unsigned)sm_count() * 4; // 4 resident CTAs of 256 threads per SM
    const int grid = (int)(p.tiles < cap ? p.tiles : cap);
    if (q.T % 2 == 0)
        return launch_overlapped(gated_residual_t_kernel<true>, grid, kResidThreads, 0, s, p);
    return launch_overlapped(gated_residual_t_kernel<false>, grid, kResidThreads, 0, s, p);
}

} // namespace dan
