/*
 * bf16_exhaustive.c -- checks the oracle's fp32 -> bf16 rounding on every one
 * of the 2^32 fp32 bit patterns (test harness; not part of the library).
 *
 * The oracle rounds by an integer add-and-shift on the bit pattern.  This
 * harness rounds a second, independent way: the two bf16 neighbours of x
 * (its truncation toward zero, and the next bf16 up in magnitude, taken as
 * 2^128 when that is the infinity pattern) are compared by their exact
 * distances to x in double arithmetic; the nearer wins, and a tie goes to the
 * neighbour with an even last bit.  That is round-to-nearest-even as IEEE 754
 * defines it, overflow to infinity included.  NaN inputs must give a NaN of the
 * same sign (their payload is not pinned).
 *
 * usage: bf16_exhaustive <path to the oracle's shared library> [threads]
 * prints "mismatches N" and exits 0 when N == 0.
 */
#include <dlfcn.h>
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

typedef void (*round_array_fn)(const uint32_t* in, uint16_t* out, size_t n);

static round_array_fn g_round;
static int g_threads;

static double value_of(uint32_t bits) {
    float f;
    memcpy(&f, &bits, 4);
    return (double)f;
}

/* Round-to-nearest-even from the two neighbours; `u` is not a NaN. */
static uint16_t nearest_bf16(uint32_t u) {
    const uint32_t sign = u & 0x80000000u, mag = u & 0x7FFFFFFFu;
    const uint32_t lo = mag & 0xFFFF0000u;
    if (lo == mag) return (uint16_t)(u >> 16);
    const uint32_t hi = lo + 0x10000u;
    const double x = value_of(mag), a = value_of(lo);
    const double b = hi == 0x7F800000u ? ldexp(1.0, 128) : value_of(hi);
    const double da = x - a, db = b - x;       /* exact: fp32 values in double */
    uint32_t pick;
    if (da < db) pick = lo;
    else if (db < da) pick = hi;
    else pick = ((lo >> 16) & 1u) == 0 ? lo : hi;
    return (uint16_t)((sign | pick) >> 16);
}

typedef struct {
    uint64_t begin, end;
    uint64_t mismatches;
    uint32_t first_bad;
} job_t;

enum { CHUNK = 1 << 20 };

static void* run(void* arg) {
    job_t* j = (job_t*)arg;
    uint32_t* in = (uint32_t*)malloc(sizeof(uint32_t) * CHUNK);
    uint16_t* out = (uint16_t*)malloc(sizeof(uint16_t) * CHUNK);
    for (uint64_t base = j->begin; base < j->end; base += CHUNK) {
        size_t n = (size_t)((j->end - base) < CHUNK ? (j->end - base) : CHUNK);
        for (size_t i = 0; i < n; i++) in[i] = (uint32_t)(base + i);
        g_round(in, out, n);
        for (size_t i = 0; i < n; i++) {
            const uint32_t u = in[i];
            const int is_nan = (u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0u;
            int ok;
            if (is_nan)
                ok = (out[i] & 0x7F80u) == 0x7F80u && (out[i] & 0x007Fu) != 0u && (out[i] >> 15) == (u >> 31);
            else
                ok = out[i] == nearest_bf16(u);
            if (!ok) {
                if (j->mismatches == 0) j->first_bad = u;
                j->mismatches++;
            }
        }
    }
    free(in);
    free(out);
    return NULL;
}

int main(int argc, char** argv) {
    if (argc < 2) {
        fprintf(stderr, "usage: %s liboracle.so [threads]\n", argv[0]);
        return 2;
    }
    void* h = dlopen(argv[1], RTLD_NOW);
    if (!h) {
        fprintf(stderr, "dlopen: %s\n", dlerror());
        return 2;
    }
    g_round = (round_array_fn)dlsym(h, "or_f32_to_bf16_rne_array");
    if (!g_round) {
        fprintf(stderr, "dlsym: %s\n", dlerror());
        return 2;
    }
    g_threads = argc > 2 ? atoi(argv[2]) : 8;
    if (g_threads < 1) g_threads = 1;
    if (g_threads > 256) g_threads = 256;
    pthread_t tid[256];
    job_t jobs[256];
    const uint64_t total = 1ull << 32, per = (total + (uint64_t)g_threads - 1) / (uint64_t)g_threads;
    for (int t = 0; t < g_threads; t++) {
        jobs[t].begin = per * (uint64_t)t;
        jobs[t].end = per * (uint64_t)(t + 1) < total ? per * (uint64_t)(t + 1) : total;
        jobs[t].mismatches = 0;
        jobs[t].first_bad = 0;
        pthread_create(&tid[t], NULL, run, &jobs[t]);
    }
    uint64_t bad = 0;
    uint32_t first = 0;
    for (int t = 0; t < g_threads; t++) {
        pthread_join(tid[t], NULL);
        if (jobs[t].mismatches && !bad) first = jobs[t].first_bad;
        bad += jobs[t].mismatches;
    }
    printf("mismatches %llu", (unsigned long long)bad);
    if (bad) printf(" first 0x%08x", first);
    printf("\n");
    return bad == 0 ? 0 : 1;
}
