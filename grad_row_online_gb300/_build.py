"""Builds libgrpo_gb300.so in-tree with nvcc for sm_103a."""
from __future__ import annotations

import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libgrpo_gb300.so")
SOURCES = ["grpo_api.cu", "grpo_prep.cu", "grpo_rows.cu", "grpo_reduce.cu",
           "grpo_logps.cu", "grpo_static.cu", "grpo_vocab.cu"]
ARCH = "-gencode=arch=compute_103a,code=sm_103a"
FLAGS = [ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xptxas", "-v"]


def compile_commands() -> list[list[str]]:
    return [["nvcc", *FLAGS, "-c", os.path.join(CSRC, s),
             "-o", os.path.join(BUILD, s.replace(".cu", ".o"))] for s in SOURCES]


def link_command() -> list[str]:
    return ["nvcc", ARCH, "-shared", *[os.path.join(BUILD, s.replace(".cu", ".o")) for s in SOURCES],
            "-o", LIB, "-lcudart"]


def build(verbose: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    procs = []
    for c in compile_commands():
        log = open(c[-1] + ".log", "w")
        procs.append((subprocess.Popen(c, stdout=log, stderr=subprocess.STDOUT), c, log))
    for p, c, log in procs:
        rc = p.wait()
        log.close()
        if rc != 0 or verbose:
            print(open(c[-1] + ".log").read())
        if rc != 0:
            raise RuntimeError("nvcc failed: " + " ".join(c))
    subprocess.run(link_command(), check=True)
    return LIB


if __name__ == "__main__":
    build(verbose=True)
