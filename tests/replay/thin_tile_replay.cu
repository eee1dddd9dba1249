// CPU replay of the register-tile thin-group kernels' plans and index arithmetic for one
// geometry and storage dtype (forward, backward-data and weight gradient, stride 1): every
// staged 16-byte copy inside its buffer and its source plane, every window and gradOutput
// read inside the staged buffer and, past the source, on a zero-filled element, every
// store inside the output and aligned for the vector stores, every output element written
// exactly once, every gradOutput position accumulated exactly once, the partial sums inside
// the workspace.  Host code only: the library source is included and the device-facing
// helpers it calls are stubbed.  Usage: thin_tile_replay <14 or 16 geometry ints> <0: bf16,
// 1: fp32>; exits non-zero and prints FAIL lines on any violation.
#include "../../bwd_gconv_fwd_gb300/csrc/thin_plane.cu"
#include <cstdio>
#include <cstdlib>
#include <vector>
namespace gconv {
int num_sms() { return 152; }
}
using namespace gconv;
static long errors = 0;
#define CHECK(cond, ...) do { if (!(cond)) { if (errors++ < 10) { printf("FAIL: " __VA_ARGS__); printf("\n"); } } } while (0)

// The staged copies of issue_rows for one buffer: (destination vector, source element or -1).
static void staged(int CG, int IH, int IW, int lo, int nrows, int nrows_max, int pitch, int pad, int64_t plane,
                   std::vector<int64_t> &src_of_vec)
{
    const int vrow = pitch / pad, vdata = IW / pad;
    const int total = CG * nrows_max * vrow;
    src_of_vec.assign(total, -1);
    const int step_r = kThinThreads / vrow, step_k = kThinThreads - step_r * vrow;
    for (int tid = 0; tid < kThinThreads; ++tid) {
        int row = tid / vrow, k = tid - row * vrow;
        for (int i = tid; i < total; i += kThinThreads) {
            const int c = CG == 1 ? 0 : row / nrows_max;
            const int j = row - c * nrows_max;
            const int ih = lo + j;
            const bool data = j < nrows && k >= 1 && k <= vdata && ih >= 0 && ih < IH;
            const int idx = row * vrow + k;
            CHECK(idx == i, "staging vector index %d != %d", idx, i);
            CHECK(idx >= 0 && idx < total, "staging vector %d outside the buffer (%d)", idx, total);
            if (data) {
                const int64_t s = c * plane + (int64_t)ih * IW + (k - 1) * pad;
                CHECK(s >= 0 && s + pad <= CG * plane, "staging source %lld outside the group's planes", (long long)s);
                if (idx >= 0 && idx < total) src_of_vec[idx] = s;
            }
            row += step_r;
            k += step_k;
            if (k >= vrow) { k -= vrow; ++row; }
        }
    }
}

int main(int argc, char **argv)
{
    int v[16];
    const int ng = argc - 2;
    if (ng == 14) {
        int a[14];
        for (int i = 0; i < 14; ++i) a[i] = atoi(argv[1 + i]);
        const int e[16] = {a[0], a[1], a[2], a[3], a[4], a[5], a[6], a[7], a[7], a[8], a[9], a[10], a[11], a[12], a[12], a[13]};
        for (int i = 0; i < 16; ++i) v[i] = e[i];
    } else if (ng == 16) {
        for (int i = 0; i < 16; ++i) v[i] = atoi(argv[1 + i]);
    } else {
        printf("usage: thin_tile_replay <14 or 16 geometry ints> <dtype 0|1>\n");
        return 2;
    }
    const int esize = atoi(argv[argc - 1]) ? 4 : 2;
    const int span_h = v[2] + v[9] + v[10] - v[13] * (v[5] - 1) - 1, span_w = v[3] + v[11] + v[12] - v[14] * (v[6] - 1) - 1;
    Geom g{v[0], v[1], v[2], v[3], v[4], v[5], v[6], v[7], v[8], v[9], v[10], v[11], v[12], v[13], v[14], v[15],
           span_h / v[7] + 1, span_w / v[8] + 1, v[1] / v[15], v[4] / v[15]};
    const gconv_pass passes[3] = {GCONV_PASS_FWD, GCONV_PASS_BWD_DATA, GCONV_PASS_BWD_WEIGHT};
    const int pad = 16 / esize;
    for (gconv_pass pass : passes) {
        ThinParams p;
        int grid = 0;
        size_t smem = 0, ws = 0;
        if (!thin_plan(g, pass, esize, &p, &grid, &smem, &ws) || !p.tile) {
            printf("pass %d: register-tile form not planned\n", (int)pass);
            continue;
        }
        const int CG = g.Cgi;
        const int nch = (p.OW + 3) / 4;
        const bool wg = pass == GCONV_PASS_BWD_WEIGHT;
        printf("pass %d: TH=%d n_strip=%d pitch=%d pl=%d pt=%d nch=%d grid=%d smem=%zu ws=%zu\n", (int)pass, p.TH,
               p.n_strip, p.pitch, p.pl, p.pt, nch, grid, smem, ws);
        CHECK(p.pl >= 0 && p.pl <= 2 && p.pt >= 0 && p.pt <= 2, "pads outside the templates");
        CHECK(p.pitch % pad == 0 && p.pitch >= pad + p.IW, "pitch");
        CHECK(smem <= (size_t)kThinSmemMax, "shared memory %zu", smem);
        const int64_t plane = (int64_t)p.IH * p.IW;
        if (!wg) {
            const int nrows_max = p.TH + 2;
            const int64_t buf_elems = (int64_t)CG * nrows_max * p.pitch;
            CHECK((size_t)(2 * buf_elems * esize) <= smem, "two buffers past the shared memory");
            const int nsub = kThinThreads / nch;
            CHECK(nsub >= 1, "no row runs");
            const int64_t out_plane = (int64_t)p.OH * p.OW, out_total = (int64_t)g.N * g.G * CG * out_plane;
            std::vector<unsigned char> written(out_total, 0);
            const bool vec = p.OW % 4 == 0;
            std::vector<int64_t> sv;
            for (int it = 0; it < g.N * g.G * p.n_strip; ++it) {
                int t = it;
                const int strip = t % p.n_strip; t /= p.n_strip;
                const int gg = t % g.G;
                const int n = t / g.G;
                const int r0 = strip * p.TH;
                const int rows = std::min(p.TH, p.OH - r0);
                staged(CG, p.IH, p.IW, r0 - p.pt, rows + 2, nrows_max, p.pitch, pad, plane, sv);
                for (int tid = 0; tid < kThinThreads; ++tid) {
                    const int chunk = tid % nch, sub = tid / nch;
                    const int c0 = chunk * 4, ncol = std::min(4, p.OW - c0);
                    const int sr = (rows + nsub - 1) / nsub, ra = sub * sr, rb = std::min(rows, ra + sr);
                    if (!(sub < nsub && ra < rb)) continue;
                    for (int r = ra; r < rb; ++r) {
                        for (int ci = 0; ci < CG; ++ci)
                            for (int a = 0; a < 3; ++a)
                                for (int k = 0; k < 6; ++k) {
                                    const int sc = pad + c0 - p.pl + k;   // staged column
                                    const int64_t e = (int64_t)(ci * nrows_max + r + a) * p.pitch + sc;
                                    CHECK(e >= 0 && e < buf_elems, "window read %lld outside the buffer", (long long)e);
                                    CHECK(r + a < rows + 2, "window row past the staged rows");
                                    // the element is the source element (r0 + r - pt + a, c0 - pl + k) or a zero
                                    const int sh = r0 + r - p.pt + a, sw = c0 - p.pl + k;
                                    const int64_t vec_i = e / pad;
                                    const int64_t s = (vec_i >= 0 && vec_i < (int64_t)sv.size()) ? sv[vec_i] : -2;
                                    const bool in_src = sh >= 0 && sh < p.IH && sw >= 0 && sw < p.IW;
                                    if (in_src) {
                                        if (k >= p.pl && k < p.pl + 4 || true)
                                            CHECK(s >= 0 && s + (e % pad) == ci * plane + (int64_t)sh * p.IW + sw,
                                                  "window element (%d,%d) not staged where read", sh, sw);
                                    } else if (sw < 0 || sw >= p.IW || sh < 0 || sh >= p.IH) {
                                        CHECK(s == -1, "padding element (%d,%d) read from a data vector", sh, sw);
                                    }
                                }
                        for (int o = 0; o < CG; ++o) {
                            const int64_t oi = (((int64_t)n * g.G + gg) * CG + o) * out_plane + (int64_t)(r0 + r) * p.OW + c0;
                            if (vec) CHECK(oi % 4 == 0, "vector store misaligned");
                            for (int j = 0; j < (vec ? 4 : ncol); ++j) {
                                CHECK(oi + j >= 0 && oi + j < out_total, "store outside the output");
                                if (oi + j >= 0 && oi + j < out_total) written[oi + j]++;
                            }
                        }
                    }
                }
            }
            for (int64_t i = 0; i < out_total; ++i) CHECK(written[i] == 1, "output %lld written %d times", (long long)i, written[i]);
            // persistent grids: each block walks a contiguous run of items, the coordinates of
            // the next item advanced by increments; they must match the divided ones and the
            // runs must cover every item once
            const int items = g.N * g.G * p.n_strip;
            for (int per_sm = 1; per_sm <= 16; per_sm *= 2) {
                const int pgrid = std::min(grid, 152 * per_sm);
                std::vector<unsigned char> cover(items, 0);
                for (int blk = 0; blk < pgrid; ++blk) {
                    const int it0 = (int)((int64_t)blk * items / pgrid), it1 = (int)((int64_t)(blk + 1) * items / pgrid);
                    int t = it0;
                    int strip = t % p.n_strip; t /= p.n_strip;
                    int gg = t % g.G, n = t / g.G;
                    for (int it = it0; it < it1; ++it) {
                        int u = it;
                        const int es = u % p.n_strip; u /= p.n_strip;
                        CHECK(strip == es && gg == u % g.G && n == u / g.G, "incremental item coordinates");
                        cover[it]++;
                        if (++strip == p.n_strip) { strip = 0; if (++gg == g.G) { gg = 0; ++n; } }
                    }
                }
                for (int i = 0; i < items; ++i) CHECK(cover[i] == 1, "item %d walked %d times", i, cover[i]);
            }
        } else {
            const int WPO = 4 / CG;
            const int nsub = (32 * WPO) / nch;
            CHECK(nsub >= 1, "no row runs");
            const int xrows_max = p.TH + 2, yrows_max = p.TH;
            const int64_t buf_elems = (int64_t)CG * (xrows_max + yrows_max) * p.pitch;
            CHECK((size_t)(2 * buf_elems * esize) <= smem, "two buffers past the shared memory");
            CHECK((size_t)grid * CG * (CG * 9 + 1) * 4 <= ws, "partial sums past the workspace");
            CHECK(grid == g.G * p.nchunk * p.n_strip, "grid");
            const int64_t yplane = (int64_t)p.OH * p.OW;
            std::vector<unsigned char> seen((int64_t)g.N * g.G * CG * yplane, 0);
            std::vector<int64_t> sx, sy;
            for (int blk = 0; blk < grid; ++blk) {
                int b = blk;
                const int strip = b % p.n_strip; b /= p.n_strip;
                const int chunkn = b % p.nchunk;
                const int gg = b / p.nchunk;
                const int r0 = strip * p.TH;
                const int rows = std::min(p.TH, p.OH - r0);
                const int n0 = chunkn * p.per_chunk, n1 = std::min(g.N, n0 + p.per_chunk);
                staged(CG, p.IH, p.IW, r0 - p.pt, rows + 2, xrows_max, p.pitch, pad, plane, sx);
                staged(CG, p.OH, p.OW, r0, rows, yrows_max, p.pitch, pad, yplane, sy);
                for (int n = n0; n < n1; ++n)
                    for (int tid = 0; tid < kThinThreads; ++tid) {
                        const int warp = tid >> 5, lane = tid & 31;
                        const int o = warp % CG, t = (warp / CG) * 32 + lane;
                        const int chunk = t % nch, sub = t / nch, c0 = chunk * 4;
                        const int sr = (rows + nsub - 1) / nsub, ra = sub * sr, rb = std::min(rows, ra + sr);
                        if (!(sub < nsub && ra < rb)) continue;
                        for (int r = ra; r < rb; ++r) {
                            for (int j = 0; j < 4; ++j) {
                                const int64_t e = (int64_t)(o * yrows_max + r) * p.pitch + pad + c0 + j;
                                CHECK(e >= 0 && e < (int64_t)CG * yrows_max * p.pitch, "gradOutput read outside");
                                const int64_t s = sy[e / pad];
                                if (c0 + j < p.OW) {
                                    CHECK(s >= 0 && s + e % pad == o * yplane + (int64_t)(r0 + r) * p.OW + c0 + j, "gradOutput element not staged");
                                    seen[(((int64_t)n * g.G + gg) * CG + o) * yplane + (int64_t)(r0 + r) * p.OW + c0 + j]++;
                                } else {
                                    CHECK(s == -1, "column past gradOutput not zero");
                                }
                            }
                            for (int ci = 0; ci < CG; ++ci)
                                for (int a = 0; a < 3; ++a)
                                    for (int k = 0; k < 6; ++k) {
                                        const int64_t e = (int64_t)(ci * xrows_max + r + a) * p.pitch + pad + c0 - p.pl + k;
                                        CHECK(e >= 0 && e < (int64_t)CG * xrows_max * p.pitch, "x window read outside");
                                        const int sh = r0 + r - p.pt + a, sw = c0 - p.pl + k;
                                        const int64_t s = sx[e / pad];
                                        if (sh >= 0 && sh < p.IH && sw >= 0 && sw < p.IW)
                                            CHECK(s >= 0 && s + e % pad == ci * plane + (int64_t)sh * p.IW + sw, "x element not staged");
                                        else
                                            CHECK(s == -1, "x padding read from a data vector");
                                    }
                        }
                    }
            }
            for (size_t i = 0; i < seen.size(); ++i) CHECK(seen[i] == 1, "gradOutput %zu accumulated %d times", i, seen[i]);
        }
    }
    printf("errors: %ld\n", errors);
    return errors ? 1 : 0;
}
