"""NVTX ranges around the C-ABI calls, observed without a GPU.

A small NVTX tool (written here in C, loaded by NVTX through NVTX_INJECTION64_PATH as a profiler
would be) logs every range push and pop.  A child process calls each entry point with an
invalid argument, which returns before any CUDA call; each call must still open and close its
range, named after the call.
"""
import os
import shutil
import subprocess
import sys
import textwrap

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

TOOL = r"""
#include <stdio.h>
#include <stdlib.h>
#include <nvtx3/nvToolsExt.h>

static FILE* g_log;
static int push_a(const char* name) { fprintf(g_log, "push %s\n", name); fflush(g_log); return 0; }
static int pop(void) { fprintf(g_log, "pop\n"); fflush(g_log); return 0; }

int InitializeInjectionNvtx2(NvtxGetExportTableFunc_t get_table) {
  const NvtxExportTableCallbacks* cb =
      (const NvtxExportTableCallbacks*)get_table(NVTX_ETID_CALLBACKS);
  NvtxFunctionTable table = 0;
  unsigned int last = 0;
  if (!cb || !cb->GetModuleFunctionTable(NVTX_CB_MODULE_CORE, &table, &last)) return 0;
  if (last < NVTX_CBID_CORE_RangePop) return 0;
  g_log = fopen(getenv("MSA_NVTX_LOG"), "w");
  if (!g_log) return 0;
  *table[NVTX_CBID_CORE_RangePushA] = (NvtxFunctionPointer)push_a;
  *table[NVTX_CBID_CORE_RangePop] = (NvtxFunctionPointer)pop;
  return 1;
}
"""

CHILD = textwrap.dedent("""
    import ctypes
    import block_sparse_long_msa_gb300 as msa
    L = msa.lib()
    bad = msa.MSA_ERR_INVALID_ARG
    n = None
    assert L.msa_index_select(n, n, n, 0, n, n, n, n, 0, n) == bad
    assert L.msa_index_select_scores(n, n, n, 0, n, n, n, n, n, 0, n) == bad
    assert L.msa_index_candidates(n, n, n, 0, n, 0, 0, n, n, n, 0, n) == bad
    assert L.msa_index_merge(n, 0, n, n, 0, n, n, n, n, 0, n) == bad
    assert L.msa_attn_prefill(n, n, n, n, 0, n, n, n, n, 0, n) == bad
    assert L.msa_attn_decode(n, n, n, n, n, n, n, 0, n) == bad
    assert L.msa_get_device_status(n, n) == bad
    fn = L.msa_attn_prefill_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_int64] + [ctypes.c_void_p] * 5
    assert fn(n, n, n, n, 0, n, n, n, n, n) == bad
""")

CALLS = ["msa_index_select", "msa_index_select_scores", "msa_index_candidates",
         "msa_index_merge", "msa_attn_prefill", "msa_attn_decode", "msa_get_device_status",
         "msa_attn_prefill_noalloc"]


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_every_call_opens_and_closes_its_range(tmp_path):
    from block_sparse_long_msa_gb300 import build
    build.build()
    src = tmp_path / "tool.c"
    src.write_text(TOOL)
    tool = tmp_path / "libtool.so"
    subprocess.run(["gcc", "-shared", "-fPIC", "-O1", "-I/usr/local/cuda/include", str(src),
                    "-o", str(tool)], check=True)
    log = tmp_path / "ranges.log"
    env = {**os.environ, "NVTX_INJECTION64_PATH": str(tool), "MSA_NVTX_LOG": str(log),
           "PYTHONPATH": ROOT, "MSA_DEBUG_CHECKS": "0"}
    r = subprocess.run([sys.executable, "-c", CHILD], env=env, cwd=ROOT, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = log.read_text().split("\n")[:-1]
    assert lines == [x for c in CALLS for x in (f"push {c}", "pop")], lines
