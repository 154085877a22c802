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
// six CTAs of 64 threads per SM; tiles of 64 channels x 64 tokens are
// numbered tokens fastest and CTA c of G takes tiles c, c + G, c + 2G, ...,
// so at any moment the CTAs stream along one band of neighbouring tiles
// (12.42 us at [1,3072,4096], against 12.56 for a contiguous run of tiles
// per CTA; running channels fastest was slower).  Both inputs of a tile
// are staged in shared memory by 16-byte asynchronous copies, one tile
// ahead: the update
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
// Other T (residual rows not 16-byte aligned): one 64-channel tile per
// CTA, each row parity on the 64 tokens whose pairs are 4-byte aligned.  The
// residual rows are staged in shared memory as 16-byte-aligned windows by
// cp.async, the products are formed on the update's channel pairs and
// stored transposed in shared memory, so the lanes of a warp take
// consecutive whole token pairs with one aligned shared load of each.
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
    int64_t n16;                      // 16-byte chunks of r (B*D*T*2 is a multiple of 16)
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

// Any T: one 64-channel tile per CTA of 128 threads (tokens fastest in the
// grid), up to kResidCtas CTAs per SM.  Residual row (b, d) starts at
// element (b*D + d)*T; D and the tile origins t0 are even, so a row starts
// on an odd element exactly when T and d are both odd.  Each row parity
// takes the 64 tokens whose pairs sit on 4-byte boundaries: [t0, t0 + 64)
// for even rows, [t0 - 1, t0 + 63) for odd ones, so inside the tensor every
// lane of a warp moves one whole aligned pair per row, and single elements
// (2-byte accesses) occur only at the ends of a residual row.  The update
// rows t0 - (T odd) .. t0 + 63 are multiplied by the gate in their own
// layout (channel pairs of one token), and the products bf16(gate * h) are
// stored transposed in shared memory, one row of 64 tokens per channel in
// that channel's token range, so lane k's pair is word k of the row
// (conflict-free).  The residual is read as 16-byte-aligned windows: for
// each channel row, the chunks from the 16-byte boundary at or before its
// segment through the segment's end (nine at most), copied by cp.async into
// shared memory before the update is loaded, so both are in flight
// together; a warp access of 4-byte words that starts off a sector boundary
// ran at about half the speed (measured).  A warp then walks channel rows
// w, w+4, ... (all of one parity): lane k takes its pair from the row's
// window (one aligned shared load, conflict-free) and its products from
// word k of the product row, and stores the pair.
__global__ void __launch_bounds__(kResidThreads, kResidCtas) gated_residual_t_kernel(const ResidParams p)
{
    constexpr int kPitchW = kTile / 2 + 1; // words per product row (32 used)
    constexpr int kRows = kTile / 4;       // channel rows per warp
    __shared__ uint32_t s_p[kTile * kPitchW + 4];
    constexpr int kWin = 9;                 // 16-byte chunks per residual window
    __shared__ uint4 s_r[kTile * kWin];     // residual windows, one per channel row
    uint16_t *s_p16 = reinterpret_cast<uint16_t *>(s_p);
    // First word of channel ch's product row; the upper 32 rows move by four
    // banks, so the eight channel octets of a transposing store hit eight
    // different bank groups.
    auto prow = [](int ch) { return ch * kPitchW + (ch >= kTile / 2 ? 4 : 0); };

    {   // L2 prefetch of the tile (it streams while the previous grid drains):
        // thread k < 64 the lines of residual row k's segment, thread 64 + k
        // those of update row t0 - 1 + k (and of row t0 + 63)
        const TileAt at = tile_at(p, blockIdx.x);
        const int64_t T = p.T, D = p.D;
        const int k = threadIdx.x & 63;
        if (threadIdx.x < 64) {
            if (at.d0 + k < D) {
                const int64_t s0 = ((int64_t)at.b * D + at.d0 + k) * T + at.t0;
                const int64_t a = s0 > 0 ? s0 - 1 : 0, z = s0 + (T - at.t0 < kTile ? T - at.t0 : kTile) - 1;
                prefetch_l2_line(p.r + a);
                prefetch_l2_line(p.r + z);
            }
        } else {
            const int nd = (int)(D - at.d0 < kTile ? D - at.d0 : kTile);
            for (int64_t t = (int64_t)at.t0 - 1 + k; t <= (int64_t)at.t0 + kTile - 1; t += 64)
                if (t >= 0 && t < T) {
                    const uint16_t *row = reinterpret_cast<const uint16_t *>(p.h) +
                                          ((int64_t)at.b * T + t) * D + at.d0;
                    prefetch_l2_line(row);
                    prefetch_l2_line(row + nd - 1);
                }
        }
    }
    grid_dependency_wait(); // no global read above this line (L2 prefetches only)
    allow_dependents();
    const int64_t T = p.T, D = p.D;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const TileAt at = tile_at(p, blockIdx.x);
    const int64_t t0 = at.t0;
    const int nd = (int)(D - at.d0 < kTile ? D - at.d0 : kTile); // channels of the tile
    const int todd = (int)(T & 1);
    const int odd = warp & todd;   // parity of this warp's rows
    const int e = 2 * lane - odd;  // this lane's pair: tokens t0 + e, t0 + e + 1
    const bool lo_ok = t0 + e >= 0 && t0 + e < T;
    const bool hi_ok = t0 + e + 1 < T;
    const int64_t rstep = 4 * T;   // elements between two rows of a warp
    const int64_t base = ((int64_t)at.b * D + at.d0 + warp) * T + t0 + e; // r[b][d0 + warp][t0 + e]

    // Residual windows: row dl's segment starts at element seg (tokens
    // t0 - parity ..; seg >= 0, since an odd row is never row 0) and its
    // window at chunk seg / 8.  B*D*T*2 is a multiple of 16, so a chunk that
    // starts inside the tensor ends inside it.  The elements of a window
    // outside its segment belong to neighbouring tiles and are never used,
    // so in place (r_out == r) their being rewritten by another CTA does not
    // matter; every element of the segment is read before this CTA writes it.
    {
        // 16 threads per row (the first kWin copy a chunk each), 8 rows per
        // pass; a thread's rows dl = tid/16 + 8i share one parity
        const int ch = tid & 15, dl0 = tid >> 4;
        int64_t seg = ((int64_t)at.b * D + at.d0 + dl0) * T + t0 - (dl0 & todd);
        const int64_t sstep = 8 * T;
#pragma unroll
        for (int i = 0; i < kTile / 8; ++i, seg += sstep) {
            const int dl = dl0 + 8 * i;
            const int64_t c16 = (seg >> 3) + ch;
            if (ch < kWin && dl < nd && c16 < p.n16) cp_async16(s_r + dl * kWin + ch, p.r + c16 * 8);
        }
        cp_async_commit();
    }

    // Products: thread (channel octet c, update rows tid/8 + 16m), update row
    // hr holding token t0 - todd + hr; D % 8 == 0, so an octet is wholly
    // inside or outside the tensor.  A token's product goes to index
    // hr - todd of an even channel's row and hr of an odd channel's.
    {
        const int c = tid & 7;
        if (8 * c < nd) {
            const int64_t dc = (int64_t)at.d0 + 8 * c;
            const uint4 g = ld_vec(reinterpret_cast<const uint4 *>(p.gate + (int64_t)at.b * p.vs + dc));
            const int64_t tb = t0 - todd;
            const int64_t hstep = 16 * (D / 8); // 16 update rows
            // chunk offset of update row tid/8 (may be negative before the
            // first pass: a pointer is formed only for rows inside the tensor)
            int64_t hoff = (((int64_t)at.b * T + tb + (tid >> 3)) * D + dc) / 8;
            constexpr int kPasses = kTile / 16 + 1;
            uint4 hv[kPasses];
#pragma unroll
            for (int m = 0; m < kPasses; ++m, hoff += hstep) {
                const int hr = (tid >> 3) + 16 * m;
                const int64_t tk = tb + hr;
                hv[m] = make_uint4(0, 0, 0, 0);
                if (hr < kTile + todd && tk >= 0 && tk < T) hv[m] = ld_stream(p.h + hoff);
            }
#pragma unroll
            for (int m = 0; m < kPasses; ++m) {
                const int hr = (tid >> 3) + 16 * m;
                if (hr >= kTile + todd) continue;
                const int ie = hr - todd, io = hr;
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    const uint32_t pr = hmul2(word(g, w), word(hv[m], w));
                    const int ch = 8 * c + 2 * w;
                    if (ie >= 0 && ie < kTile) s_p16[2 * prow(ch) + ie] = (uint16_t)pr;
                    if (io < kTile) s_p16[2 * prow(ch + 1) + io] = (uint16_t)(pr >> 16);
                }
            }
        }
    }
    cp_async_wait_all(); // this thread's window chunks; the barrier publishes everyone's
    __syncthreads();

    uint16_t *q = p.r_out + base;
    const uint32_t *s_r32 = reinterpret_cast<const uint32_t *>(s_r);
    // window offset (in words) of this lane's pair: rows of a warp are 4T
    // elements apart, so the segment's position in its 16-byte chunk
    // alternates between two values when T is odd and is fixed otherwise
    const int mis0 = (int)((base - 2 * lane) & 7); // even: 0, 2, 4 or 6
    const int w0 = (mis0 >> 1) + lane, w1 = ((mis0 ^ (4 * todd)) >> 1) + lane;
#pragma unroll
    for (int j = 0; j < kRows; ++j, q += rstep) {
        const int dl = warp + 4 * j;
        if (dl >= nd) break; // warp-uniform
        const uint32_t r2 = s_r32[dl * (4 * kWin) + ((j & 1) ? w1 : w0)]; // tokens t0 + e, + 1
        const uint32_t v = hadd2(r2, s_p[prow(dl) + lane]);
        if (lo_ok && hi_ok) *reinterpret_cast<uint32_t *>(q) = v;
        else if (lo_ok) q[0] = (uint16_t)v;
        else if (hi_ok) q[1] = (uint16_t)(v >> 16);
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

// CTA c takes tiles c, c + G, c + 2G, ...  Requires T % 8 == 0.
__global__ void __launch_bounds__(kPThreads, kPipeCtas) gated_residual_t_pipe_kernel(const ResidParams p)
{
    extern __shared__ __align__(128) uint4 s_pipe[]; // kStages x (update, residual)
    const unsigned G = gridDim.x;
    const unsigned first = blockIdx.x; // tiles first + G * i
    const unsigned n = (p.tiles - first + G - 1) / G;
    // L2 prefetch of the first tiles (they stream while the previous grid
    // drains): thread k takes update row k and residual row k of each tile.
    for (unsigned i = 0; i < (unsigned)(kStages - 1) && i < n; ++i) {
        const PipeTile at = pipe_tile(p, first + G * i);
        const int k = threadIdx.x;
        const int64_t T = p.T, D = p.D;
        const int64_t nd = D - at.d0 < kPD ? D - at.d0 : kPD, nt = T - at.t0 < kPT ? T - at.t0 : kPT;
        if (k < nt)
            prefetch_l2(p.h + (((int64_t)at.b * T + at.t0 + k) * D + at.d0) / 8, (unsigned)nd * 2u);
        if (k < nd)
            prefetch_l2(p.r + ((int64_t)at.b * D + at.d0 + k) * T + at.t0, (unsigned)nt * 2u);
    }
    grid_dependency_wait(); // no global read above this line (L2 prefetches only)
    allow_dependents();
    auto tile_of = [&](unsigned i) { return first + G * i; };
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
    p.n16 = q.B * q.D * q.T / 8;
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
