/*
 * oracle/tile_model.c -- counting model of one shared-memory tile scan:
 * how many adds the Hillis-Steele and Blelloch trees make, and how many
 * warp-wide shared-memory requests each tree level costs once bank
 * conflicts split it.
 *
 * TEST INFRASTRUCTURE ONLY (see scan_ref.c); the CUDA library never uses it.
 *
 * Source: "The CUDA scan algorithm: the tree and the three kernels",
 * sections "Two sweeps over one tree", "The stride doubles, and so does the
 * conflict" and the "Tile model, computed at compile time" table in Results.
 * The model counts, it does not time:
 *
 *   - Blelloch level `stride` (1, 2, 4, ... < tile) makes tile/(2*stride)
 *     adds; add k touches words a = (2k+1)*stride - 1 and
 *     b = (2k+2)*stride - 1.  The down-sweep repeats the same levels.
 *   - Hillis-Steele step `offset` (1, 2, 4, ... < tile): element i >= offset
 *     adds element i - offset.
 *   - Adds are handed to lanes in order, 32 to a warp (k = 32w .. 32w+31).
 *   - A warp's request count for one access is the largest number of
 *     distinct 32-bit words that fall in one of the 32 banks (word w sits in
 *     bank w mod 32; lanes reading the same word share it).
 *   - Padding maps logical word i to i + i/32 (one term) or
 *     i + i/32 + i/1024 (two terms) ("The stride doubles ..." and the
 *     bank-padding formula phys = logical + (logical >> 5) of "Parallel
 *     Prefix Sum (Scan) for NVIDIA T4 (sm_75)", Key Features).
 *
 * Reading: the page counts one request set per warp per level, whose size is
 * the larger of the two accesses' conflict degrees (a and b); the per-tile
 * total sums that over every level of both sweeps.
 */
#include <stdint.h>

enum { LAYOUT_PLAIN = 0, LAYOUT_PAD32 = 1, LAYOUT_PAD32_1024 = 2 };

static uint64_t padded_word(uint64_t i, int layout)
{
    if (layout == LAYOUT_PAD32)
        return i + i / 32;
    if (layout == LAYOUT_PAD32_1024)
        return i + i / 32 + i / 1024;
    return i;
}

/* Largest number of distinct words that share one bank among `cnt` words. */
static int bank_degree(const uint64_t *words, int cnt)
{
    int worst = 0;
    for (int bank = 0; bank < 32; ++bank) {
        int distinct = 0;
        for (int i = 0; i < cnt; ++i) {
            if (words[i] % 32 != (uint64_t)bank)
                continue;
            int seen = 0;
            for (int j = 0; j < i; ++j)
                if (words[j] == words[i])
                    seen = 1;
            if (!seen)
                distinct += 1;
        }
        if (distinct > worst)
            worst = distinct;
    }
    return worst;
}

/* Adds made by the Blelloch up-sweep plus down-sweep over `tile` words. */
uint64_t oracle_blelloch_adds(uint64_t tile)
{
    uint64_t adds = 0;
    for (uint64_t stride = 1; stride < tile; stride *= 2)
        adds += tile / (2 * stride); /* up-sweep level */
    for (uint64_t stride = tile / 2; stride > 0; stride /= 2)
        adds += tile / (2 * stride); /* down-sweep level: one add per swap */
    return adds;
}

/* Adds made by the Hillis-Steele scan over `n` elements. */
uint64_t oracle_hillis_steele_adds(uint64_t n)
{
    uint64_t adds = 0;
    for (uint64_t offset = 1; offset < n; offset *= 2)
        for (uint64_t i = offset; i < n; ++i)
            adds += 1;
    return adds;
}

/* Number of warp passes at Blelloch level `stride` over `tile` words. */
int oracle_blelloch_level_warps(uint64_t tile, uint64_t stride)
{
    uint64_t adds = tile / (2 * stride);
    return (int)((adds + 31) / 32);
}

/*
 * Worst conflict degree over the warps of Blelloch level `stride`, for the
 * given layout.  Each warp's degree is the larger of its a- and b-access
 * degrees.
 */
int oracle_blelloch_level_degree(uint64_t tile, uint64_t stride, int layout)
{
    uint64_t adds = tile / (2 * stride);
    int worst = 0;
    for (uint64_t w = 0; w * 32 < adds; ++w) {
        uint64_t wa[32], wb[32];
        int cnt = 0;
        for (uint64_t k = w * 32; k < adds && k < w * 32 + 32; ++k) {
            wa[cnt] = padded_word((2 * k + 1) * stride - 1, layout);
            wb[cnt] = padded_word((2 * k + 2) * stride - 1, layout);
            cnt += 1;
        }
        int da = bank_degree(wa, cnt);
        int db = bank_degree(wb, cnt);
        int d = da > db ? da : db;
        if (d > worst)
            worst = d;
    }
    return worst;
}

/* Requests per tile for the Blelloch tree: both sweeps, every level. */
uint64_t oracle_blelloch_requests(uint64_t tile, int layout)
{
    uint64_t total = 0;
    for (uint64_t stride = 1; stride < tile; stride *= 2) {
        uint64_t adds = tile / (2 * stride);
        uint64_t level = 0;
        for (uint64_t w = 0; w * 32 < adds; ++w) {
            uint64_t wa[32], wb[32];
            int cnt = 0;
            for (uint64_t k = w * 32; k < adds && k < w * 32 + 32; ++k) {
                wa[cnt] = padded_word((2 * k + 1) * stride - 1, layout);
                wb[cnt] = padded_word((2 * k + 2) * stride - 1, layout);
                cnt += 1;
            }
            int da = bank_degree(wa, cnt);
            int db = bank_degree(wb, cnt);
            level += (uint64_t)(da > db ? da : db);
        }
        total += 2 * level; /* the down-sweep walks the same level */
    }
    return total;
}

/* Requests per tile for the Hillis-Steele scan over `tile` words. */
uint64_t oracle_hillis_steele_requests(uint64_t tile)
{
    uint64_t total = 0;
    for (uint64_t offset = 1; offset < tile; offset *= 2) {
        for (uint64_t w = 0; w * 32 < tile; ++w) {
            uint64_t words[32];
            int cnt = 0;
            for (uint64_t t = w * 32; t < tile && t < w * 32 + 32; ++t)
                words[cnt++] = t;
            total += (uint64_t)bank_degree(words, cnt);
        }
    }
    return total;
}
