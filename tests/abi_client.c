/*
 * A plain C99 client of include/demo.h, built and run by tests/test_c_client.py.
 *
 * It shows that the header is valid C (no C++ types or keywords leak through
 * the extern "C" block) and that a C program links against the library and
 * calls its host-only entry points: status names, payload sizes, the payload
 * validator, the argument checks of the multi-replica encode, and the device
 * probe.  It prints one "key value" line per result; the Python side compares
 * them with the oracle's payload sizes and with the header's stated
 * conventions.  No call here launches a kernel.
 */
#include <stdio.h>
#include <stdint.h>
#include <string.h>

#include "demo.h"

static void print_sizes(const char* tag, int mode, int64_t n, int k, uint64_t step) {
  size_t idx = 12345;
  size_t vals = demo_payload_bytes(mode, n, DEMO_CHUNK, k, step, 8, &idx);
  printf("%s %lu %lu\n", tag, (unsigned long)vals, (unsigned long)idx);
}

int main(void) {
  int codes[7] = {DEMO_OK, DEMO_EINVAL, DEMO_EALIGN, DEMO_ENODEV, DEMO_ECUDA, DEMO_ENOTINIT, DEMO_ENOSPACE};
  int i;
  uint8_t idx[4 * 3];
  int64_t bad = -7;
  unsigned int fault = 0;
  int init, rc;

  for (i = 0; i < 7; ++i) printf("status %d %s\n", codes[i], demo_status_string(codes[i]));

  print_sizes("demo_k4", DEMO_MODE_DEMO, 32 * 1000, 4, 0);
  print_sizes("random_k8", DEMO_MODE_RANDOM, 32 * 1000, 8, 0);
  print_sizes("stride_k4", DEMO_MODE_STRIDE, 32 * 1000, 4, 0);
  print_sizes("diloco_s6", DEMO_MODE_DILOCO, 32 * 1000, 1, 6);
  print_sizes("diloco_s7", DEMO_MODE_DILOCO, 32 * 1000, 1, 7);
  print_sizes("bad_n", DEMO_MODE_DEMO, 48, 4, 0);
  printf("ternary_k4 %lu\n",
         (unsigned long)demo_payload_bytes_wire(DEMO_MODE_DEMO, 32 * 1000, DEMO_CHUNK, 4, 0, 8, DEMO_WIRE_TERNARY,
                                                NULL));

  /* three chunks of k = 4 ascending, distinct indices in [0, 32) */
  for (i = 0; i < 3; ++i) {
    idx[4 * i + 0] = 0;
    idx[4 * i + 1] = 5;
    idx[4 * i + 2] = 17;
    idx[4 * i + 3] = 31;
  }
  printf("validate_ok %d\n", demo_validate_payload(3 * DEMO_CHUNK, DEMO_CHUNK, 4, DEMO_WIRE_F32, idx, &bad));
  idx[4 * 2 + 2] = 5; /* chunk 2 repeats index 5 */
  rc = demo_validate_payload(3 * DEMO_CHUNK, DEMO_CHUNK, 4, DEMO_WIRE_F32, idx, &bad);
  printf("validate_dup %d %ld\n", rc, (long)bad);
  idx[4 * 2 + 2] = 17;
  idx[4 * 1 + 3] = 32; /* chunk 1 holds an index past the chunk */
  rc = demo_validate_payload(3 * DEMO_CHUNK, DEMO_CHUNK, 4, DEMO_WIRE_F32, idx, &bad);
  printf("validate_range %d %ld\n", rc, (long)bad);

  {
    /* demo_encode_replicas refuses before any launch: no replicas, and two replicas sharing one
       momentum buffer (the addresses are never dereferenced) */
    const void* g[2];
    float* m[2];
    void* v[2];
    void* ix[2];
    g[0] = (const void*)(uintptr_t)0x100000u;
    g[1] = (const void*)(uintptr_t)0x200000u;
    m[0] = (float*)(uintptr_t)0x1000000u;
    m[1] = (float*)(uintptr_t)0x1000000u;
    v[0] = (void*)(uintptr_t)0x30000u;
    v[1] = (void*)(uintptr_t)0x31000u;
    ix[0] = (void*)(uintptr_t)0x32000u;
    ix[1] = (void*)(uintptr_t)0x33000u;
    rc = demo_encode_replicas(g, DEMO_GRAD_F32, m, 64, DEMO_CHUNK, 4, 0.9f, DEMO_MODE_DEMO, 1, 0, 8, 0, 0,
                              DEMO_WIRE_F32, v, ix, NULL);
    printf("replicas_none %d\n", rc);
    rc = demo_encode_replicas(g, DEMO_GRAD_F32, m, 64, DEMO_CHUNK, 4, 0.9f, DEMO_MODE_DEMO, 1, 2, 8, 0, 0,
                              DEMO_WIRE_F32, v, ix, NULL);
    printf("replicas_shared_m %d\n", rc);
  }

  init = demo_init(0);
  printf("init %d\n", init);
  rc = demo_device_fault(&fault);
  printf("fault %d %u\n", rc, fault);
  return 0;
}
