/*
 * Seeded synthetic inputs for the sparse voxel-grid stencil pipeline.
 *
 * This file is shared by the CPU oracle and the CUDA path: it only makes
 * inputs (active-voxel coordinate sets and per-voxel sidecar values).  It holds
 * none of the pipeline's arithmetic (no tree order, no indexing, no stencil),
 * so both sides can use it without sharing any of the method's code.
 *
 * Randomness is counter based: value k of stream `seed` is SplitMix64's output
 * mix (Steele, Lea & Flood, "Fast splittable pseudorandom number generators",
 * OOPSLA 2014) applied to seed ^ (k * golden gamma).  Only integer arithmetic
 * and plain double arithmetic (no libm) decide which voxels are active, so the
 * coordinate sets are identical on every machine when compiled with
 * -ffp-contract=off.
 */
#include <stdint.h>
#include <stddef.h>
#include <math.h>
#include <stdlib.h>

#define GOLDEN 0x9E3779B97F4A7C15ULL

static uint64_t mix64(uint64_t z) {
    z += GOLDEN;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

uint64_t synth_hash64(uint64_t seed, uint64_t k) { return mix64(seed ^ (k * GOLDEN)); }

/* 53-bit uniform in [0,1). */
static double unit53(uint64_t h) { return (double)(h >> 11) * (1.0 / 9007199254740992.0); }

/* Stream separators so that different draws never reuse a counter. */
#define STREAM_LEAF_ON   0x6C6561666F6E0001ULL
#define STREAM_LEAF_RHO  0x6C656166726F0002ULL
#define STREAM_LEAF_BIT  0x6C65616662690003ULL
#define STREAM_LEAF_FORCE 0x6C65616666720004ULL
#define STREAM_FOG       0x666F676C61740005ULL
#define STREAM_NORMAL    0x6E6F726D616C0006ULL
#define STREAM_SCATTER   0x7363617474720007ULL

/* ---------------------------------------------------------------------------
 * Sidecars: (n+1) rows of C floats, row r at out[r*C .. r*C+C-1]; row 0 = 0.
 * ------------------------------------------------------------------------- */

/* U[-1,1): 24 random bits mapped to (int)u24 - 2^23, times 2^-23 (exact). */
void synth_sidecar_uniform(uint64_t seed, int64_t n, int C, float* out) {
    for (int c = 0; c < C; ++c) out[c] = 0.0f;
    for (int64_t r = 1; r <= n; ++r) {
        for (int c = 0; c < C; ++c) {
            uint64_t k = (uint64_t)r * (uint64_t)C + (uint64_t)c;
            int32_t u24 = (int32_t)(synth_hash64(seed, k) >> 40);
            out[r * C + c] = (float)(u24 - 8388608) * (1.0f / 8388608.0f);
        }
    }
}

/* N(0,1) by Box-Muller from two 53-bit uniforms, rounded to float. */
void synth_sidecar_normal(uint64_t seed, int64_t n, int C, float* out) {
    const double two_pi = 6.283185307179586476925286766559;
    for (int c = 0; c < C; ++c) out[c] = 0.0f;
    for (int64_t r = 1; r <= n; ++r) {
        for (int c = 0; c < C; ++c) {
            uint64_t k = (uint64_t)r * (uint64_t)C + (uint64_t)c;
            double u1 = unit53(synth_hash64(seed ^ STREAM_NORMAL, 2 * k)) + (1.0 / 9007199254740992.0);
            double u2 = unit53(synth_hash64(seed ^ STREAM_NORMAL, 2 * k + 1));
            out[r * C + c] = (float)(sqrt(-2.0 * log(u1)) * cos(two_pi * u2));
        }
    }
}

/* ---------------------------------------------------------------------------
 * Coordinate sets.  Each returns the number of active voxels; it writes at most
 * `cap` coordinate triples (x,y,z int32) into `out` (which may be NULL to count).
 * ------------------------------------------------------------------------- */

/* Sphere shell about the origin: integer points with r_in <= |p| <= r_out. */
int64_t synth_shell(double r_in, double r_out, int32_t* out, int64_t cap) {
    int64_t n = 0;
    int32_t R = (int32_t)ceil(r_out) + 1;
    double lo = r_in * r_in, hi = r_out * r_out;
    for (int32_t x = -R; x <= R; ++x)
        for (int32_t y = -R; y <= R; ++y)
            for (int32_t z = -R; z <= R; ++z) {
                double d2 = (double)((int64_t)x * x + (int64_t)y * y + (int64_t)z * z);
                if (d2 >= lo && d2 <= hi) {
                    if (out && n < cap) { out[3 * n] = x; out[3 * n + 1] = y; out[3 * n + 2] = z; }
                    ++n;
                }
            }
    return n;
}

/* Random 8^3 bricks: a cube of dim_b^3 bricks at the origin; each brick is on
 * with probability p_on; an on brick draws a density rho ~ U[rho_lo, rho_hi) and
 * turns each of its 512 cells on with probability rho (at least one forced). */
int64_t synth_bricks(int dim_b, double p_on, double rho_lo, double rho_hi, uint64_t seed,
                     int32_t* out, int64_t cap) {
    int64_t n = 0;
    for (int bi = 0; bi < dim_b; ++bi)
        for (int bj = 0; bj < dim_b; ++bj)
            for (int bk = 0; bk < dim_b; ++bk) {
                uint64_t lin = ((uint64_t)bi * dim_b + bj) * dim_b + bk;
                if (!(unit53(synth_hash64(seed ^ STREAM_LEAF_ON, lin)) < p_on)) continue;
                double rho = rho_lo + (rho_hi - rho_lo) * unit53(synth_hash64(seed ^ STREAM_LEAF_RHO, lin));
                int any = 0;
                int forced = (int)(synth_hash64(seed ^ STREAM_LEAF_FORCE, lin) % 512u);
                for (int a = 0; a < 8; ++a)
                    for (int b = 0; b < 8; ++b)
                        for (int c = 0; c < 8; ++c) {
                            int cell = (a * 8 + b) * 8 + c;
                            int on = unit53(synth_hash64(seed ^ STREAM_LEAF_BIT, lin * 512u + (uint64_t)cell)) < rho;
                            if (on) {
                                any = 1;
                                if (out && n < cap) {
                                    out[3 * n] = bi * 8 + a; out[3 * n + 1] = bj * 8 + b; out[3 * n + 2] = bk * 8 + c;
                                }
                                ++n;
                            }
                        }
                if (!any) {
                    int a = forced / 64, b = (forced / 8) % 8, c = forced % 8;
                    if (out && n < cap) {
                        out[3 * n] = bi * 8 + a; out[3 * n + 1] = bj * 8 + b; out[3 * n + 2] = bk * 8 + c;
                    }
                    ++n;
                }
            }
    return n;
}

/* Fog: fractal value noise on [0,dim)^3.  Octave o has period P_o = 64 >> o
 * (o = 0..3) and amplitude 2^-o; the lattice value at integer lattice point
 * (a,b,c) is a U[0,1) draw keyed by (o,a,b,c); the field at voxel (i,j,k) is the
 * trilinear interpolation at ((i+.5)/P, (j+.5)/P, (k+.5)/P), interpolated along
 * x, then y, then z (lerp(u,v,t) = u + (v-u)*t in double).  The octaves are
 * summed and divided by 1.875; a voxel is active iff the result > threshold.
 * Writes one byte per voxel (x-major: mask[(i*dim+j)*dim+k]) and returns the
 * count.  dim must be a multiple of 64. */
static double lerp_d(double u, double v, double t) { return u + (v - u) * t; }

int64_t synth_fog_mask(int dim, uint64_t seed, double threshold, uint8_t* mask) {
    enum { NOCT = 4 };
    const int period[NOCT] = {64, 32, 16, 8};
    const double amp[NOCT] = {1.0, 0.5, 0.25, 0.125};
    int ext[NOCT];
    double* lat[NOCT];
    double* row[NOCT];
    int64_t n = 0;
    if (dim <= 0 || dim % 64) return -1;
    for (int o = 0; o < NOCT; ++o) {
        ext[o] = dim / period[o] + 1;
        int e = ext[o];
        lat[o] = (double*)malloc(sizeof(double) * (size_t)e * e * e);
        row[o] = (double*)malloc(sizeof(double) * (size_t)e);
        for (int a = 0; a < e; ++a)
            for (int b = 0; b < e; ++b)
                for (int c = 0; c < e; ++c) {
                    uint64_t key = (((uint64_t)o * 4096u + (uint64_t)a) * 4096u + (uint64_t)b) * 4096u + (uint64_t)c;
                    lat[o][((size_t)a * e + b) * e + c] = unit53(synth_hash64(seed ^ STREAM_FOG, key));
                }
    }
    for (int i = 0; i < dim; ++i)
        for (int j = 0; j < dim; ++j) {
            for (int o = 0; o < NOCT; ++o) {
                int e = ext[o];
                double ux = ((double)i + 0.5) / period[o], uy = ((double)j + 0.5) / period[o];
                int ax = (int)floor(ux), ay = (int)floor(uy);
                double fx = ux - ax, fy = uy - ay;
                const double* l = lat[o];
                for (int c = 0; c < e; ++c) {
                    double v00 = lerp_d(l[((size_t)ax * e + ay) * e + c], l[((size_t)(ax + 1) * e + ay) * e + c], fx);
                    double v01 = lerp_d(l[((size_t)ax * e + ay + 1) * e + c], l[((size_t)(ax + 1) * e + ay + 1) * e + c], fx);
                    row[o][c] = lerp_d(v00, v01, fy);
                }
            }
            for (int k = 0; k < dim; ++k) {
                double s = 0.0;
                for (int o = 0; o < NOCT; ++o) {
                    double uz = ((double)k + 0.5) / period[o];
                    int az = (int)floor(uz);
                    double fz = uz - az;
                    s += amp[o] * lerp_d(row[o][az], row[o][az + 1], fz);
                }
                s /= 1.875;
                uint8_t on = s > threshold;
                mask[((size_t)i * dim + j) * dim + k] = on;
                n += on;
            }
        }
    for (int o = 0; o < NOCT; ++o) { free(lat[o]); free(row[o]); }
    return n;
}

/* Coordinates of the set cells of a dim^3 byte mask, x-major. */
int64_t synth_mask_coords(const uint8_t* mask, int dim, int32_t* out, int64_t cap) {
    int64_t n = 0;
    for (int i = 0; i < dim; ++i)
        for (int j = 0; j < dim; ++j)
            for (int k = 0; k < dim; ++k)
                if (mask[((size_t)i * dim + j) * dim + k]) {
                    if (out && n < cap) { out[3 * n] = i; out[3 * n + 1] = j; out[3 * n + 2] = k; }
                    ++n;
                }
    return n;
}

/* Scatter: `count` distinct points, each the single active cell of its own
 * 8-aligned brick: brick b sits at 8*(b_x, b_y, b_z) with b on a cube of side
 * `side` bricks (count <= side^3), stepping through bricks in a seeded
 * permutation-free order (every brick, raster order, first `count`), and the
 * cell inside the brick is drawn at random.  `origin` shifts every point. */
int64_t synth_scatter(int side, int64_t count, int32_t origin, uint64_t seed, int32_t* out, int64_t cap) {
    int64_t n = 0;
    for (int64_t b = 0; b < (int64_t)side * side * side && n < count; ++b) {
        int bx = (int)(b / ((int64_t)side * side)), by = (int)((b / side) % side), bz = (int)(b % side);
        uint64_t h = synth_hash64(seed ^ STREAM_SCATTER, (uint64_t)b);
        int cx = (int)(h & 7), cy = (int)((h >> 3) & 7), cz = (int)((h >> 6) & 7);
        if (out && n < cap) {
            out[3 * n] = origin + bx * 8 + cx; out[3 * n + 1] = origin + by * 8 + cy; out[3 * n + 2] = origin + bz * 8 + cz;
        }
        ++n;
    }
    return n;
}
