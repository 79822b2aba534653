"""The extension build's rebuild decisions (CPU only; the compiler is faked).

build() recompiles an object when its content key (source, every header,
flags, compiler id, machine type) differs from the one recorded beside it,
and relinks the library when any object key changed. These tests drive it on
a throwaway source tree with a stand-in for nvcc that records what it was
asked to compile and writes placeholder outputs.
"""
import importlib.util
import os
import time

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture
def tree(tmp_path, monkeypatch):
    spec = importlib.util.spec_from_file_location(
        "build_under_test", os.path.join(ROOT, "ulysses_sequence_attention_gb300", "build.py"))
    b = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(b)
    pkg, inc = tmp_path / "pkg", tmp_path / "include"
    (pkg / "csrc").mkdir(parents=True)
    inc.mkdir()
    (pkg / "csrc" / "a.cu").write_text("// a\n")
    (pkg / "csrc" / "b.cu").write_text("// b\n")
    (pkg / "csrc" / "common.cuh").write_text("// common\n")
    (inc / "api.h").write_text("// api\n")
    monkeypatch.setattr(b, "CSRC", str(pkg / "csrc"))
    monkeypatch.setattr(b, "INCLUDE", str(inc))
    monkeypatch.setattr(b, "BUILD_DIR", str(pkg / "_build"))
    monkeypatch.setattr(b, "LIB_PATH", str(pkg / "libulysses.so"))
    monkeypatch.setattr(b, "_nvcc", lambda: "nvcc")
    monkeypatch.setattr(b, "_compiler_id", lambda nvcc: "nvcc 13.0 (stand-in)")
    log = {"compiled": [], "linked": 0}

    class Done:
        returncode, stdout, stderr = 0, "", ""

    def fake_run(cmd, capture_output=True, text=True):
        out = cmd[cmd.index("-o") + 1]
        if "-c" in cmd:
            log["compiled"].append(os.path.basename(cmd[cmd.index("-c") + 1]))
        else:
            log["linked"] += 1
        with open(out, "w") as f:
            f.write("built\n")
        return Done()

    monkeypatch.setattr(b.subprocess, "run", fake_run)

    def build():
        log["compiled"], log["linked"] = [], 0
        b.build()
        return sorted(log["compiled"]), log["linked"]

    return b, pkg, inc, build


def test_first_build_compiles_everything_and_a_second_build_nothing(tree):
    b, pkg, inc, build = tree
    assert build() == (["a.cu", "b.cu"], 1)
    assert build() == ([], 0)


def test_a_newer_file_time_alone_rebuilds_nothing(tree):
    b, pkg, inc, build = tree
    build()
    later = time.time() + 100
    for p in (pkg / "csrc" / "a.cu", inc / "api.h"):
        os.utime(p, (later, later))
    assert build() == ([], 0)


def test_a_changed_source_rebuilds_that_object_and_relinks(tree):
    b, pkg, inc, build = tree
    build()
    (pkg / "csrc" / "b.cu").write_text("// b, edited\n")
    assert build() == (["b.cu"], 1)


@pytest.mark.parametrize("header", ["csrc/common.cuh", "api.h"])
def test_a_changed_header_rebuilds_every_object(tree, header):
    b, pkg, inc, build = tree
    build()
    path = (pkg / header) if header.startswith("csrc") else (inc / header)
    path.write_text("// edited\n")
    assert build() == (["a.cu", "b.cu"], 1)


def test_a_foreign_object_newer_than_its_source_is_not_reused(tree):
    b, pkg, inc, build = tree
    build()
    # a binary copied in from elsewhere, with a key that is not this tree's
    (pkg / "_build" / "a.o").write_text("foreign\n")
    (pkg / "_build" / "a.key").write_text("0" * 64 + "\n")
    assert build() == (["a.cu"], 1)


def test_a_missing_key_or_library_is_rebuilt(tree):
    b, pkg, inc, build = tree
    build()
    os.unlink(pkg / "_build" / "b.key")
    assert build() == (["b.cu"], 1)
    os.unlink(pkg / "libulysses.so")
    assert build() == ([], 1)
    (pkg / "_build" / "libulysses.key").write_text("stale\n")
    assert build() == ([], 1)


def test_flags_are_part_of_the_key(tree, monkeypatch):
    b, pkg, inc, build = tree
    build()
    monkeypatch.setattr(b, "NVCC_FLAGS", b.NVCC_FLAGS + ["-DEXTRA"])
    assert build() == (["a.cu", "b.cu"], 1)
