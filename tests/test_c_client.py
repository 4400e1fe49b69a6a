"""The boundary from plain C: a C11 program includes include/das.h, links
libdas.so and makes calls that the library answers on the host (version,
rejected arguments, the thread's error text).  Needs gcc and the CUDA headers
(for cudaStream_t), no GPU."""
import os
import shutil
import subprocess
from pathlib import Path

import pytest

from volumetric_ultrasound_delay_gb300 import build as build_mod

ROOT = Path(__file__).resolve().parent.parent

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "das.h"

int main(void)
{
    das_plan plan = NULL;
    const float rx[3] = {0.f, 0.f, 0.f};
    das_grid bad = {0, 4, 4, 0.f, 0.f, 0.01f, 1e-3f, 1e-3f, 1e-3f, NULL};
    int fails = 0;
    printf("version %s\n", das_version());
    /* a NULL plan handle, then a grid with nx = 0: rejected before any device call */
    if (das_plan_create(NULL, &bad, rx, 1540.f, 20e6f, 0.f, 1.5f, DAS_F32, 1, 1, 1, 8) != DAS_ERR_INVALID_ARG) fails++;
    if (das_plan_create(&plan, &bad, rx, 1540.f, 20e6f, 0.f, 1.5f, DAS_F32, 1, 1, 1, 8) != DAS_ERR_INVALID_ARG) fails++;
    if (plan != NULL) fails++;
    if (strlen(das_last_error_string()) == 0) fails++;
    printf("error %s\n", das_last_error_string());
    if (das_beamform(NULL, NULL, NULL, NULL, NULL, 0) != DAS_ERR_INVALID_ARG) fails++;
    if (das_permute(NULL, NULL, DAS_F32, 1, 1, 1, 1, 0, DAS_STORAGE_NATIVE, 0) != DAS_ERR_INVALID_ARG) fails++;
    if (das_plan_destroy(NULL) != DAS_OK) fails++;
    printf("fails %d\n", fails);
    return fails;
}
"""


def _cuda_include():
    nvcc = Path(build_mod.nvcc()).resolve()
    inc = nvcc.parent.parent / "include"
    return inc if (inc / "cuda_runtime_api.h").exists() else None


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_c_program_compiles_links_and_gets_host_answers(tmp_path):
    lib = build_mod.build()
    inc = _cuda_include()
    if inc is None:
        pytest.skip("CUDA headers not found")
    src = tmp_path / "client.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "client"
    subprocess.run(["gcc", "-std=c11", "-Wall", "-Werror", "-I", str(ROOT / "include"), "-I", str(inc),
                    str(src), "-o", str(exe), "-L", str(Path(lib).parent), "-ldas",
                    f"-Wl,-rpath,{Path(lib).parent}"], check=True)
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    out = subprocess.run([str(exe)], capture_output=True, text=True, env=env, timeout=60)
    assert out.returncode == 0, out.stdout + out.stderr
    assert "version 1.0.0" in out.stdout and "fails 0" in out.stdout
    assert "grid dimensions" in out.stdout
