"""Host logic of bench.py that needs no GPU: the extension table of the
single-workload mode builds caches the library accepts, the byte counts of
each storage variant, and the single-GPU guard of --case."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from bit_kv_cache_06_gb300 import build as kbuild  # noqa: E402
from bit_kv_cache_06_gb300 import kivi, synth  # noqa: E402


@pytest.fixture(scope="module")
def L():
    kbuild.build()
    return kivi.load()


@pytest.mark.parametrize("name", sorted(bench.EXTENSIONS))
def test_every_extension_is_a_valid_cache_on_the_8b_layer(L, name):
    w, var = bench.extension_case(synth.C2, name)
    shape = kivi.CacheShape(w.bits, w.G, w.R, w.B, w.Hq, w.Hkv, w.d, w.capacity(), **var)
    assert kivi.params_validate(shape.params()) == kivi.KIVI_OK
    assert (w.B, w.Hq, w.Hkv, w.T) == (synth.C2.B, synth.C2.Hq, synth.C2.Hkv, synth.C2.T)


def test_extension_case_copies_its_fields():
    _, a = bench.extension_case(synth.C2, "sink-4")
    a["sink_tokens"] = 99
    _, b = bench.extension_case(synth.C2, "sink-4")
    assert b == {"sink_tokens": 4}


def test_bytes_per_token_pair_of_each_storage():
    # 2-bit G = 32 d = 128: 64 B of codes + 32 B key and 32 B value metadata
    # (fp32), half of that metadata in fp16; FP8 one byte per element
    assert bench.bytes_per_quant_token(2, 32, 128, meta=0) == 128
    assert bench.bytes_per_quant_token(2, 32, 128, meta=1) == 96
    assert bench.bytes_per_quant_token(4, 64, 128, meta=0) == 160
    assert bench.bytes_per_quant_token(4, 32, 128, meta=0) == 192
    assert bench.bytes_per_quant_token(8, 32, 128) == 256


def test_case_mode_refuses_several_ranks(monkeypatch):
    monkeypatch.setenv("RANK", "0")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setattr(sys, "argv", ["bench.py", "--gpus", "2", "--case", "c2"])
    called = []
    monkeypatch.setattr(bench, "run_case", lambda args: called.append(args) or {})
    monkeypatch.setattr(bench.torch.distributed, "init_process_group",
                        lambda *a, **k: pytest.fail("no process group for --case"))
    with pytest.raises(SystemExit) as e:
        bench.main()
    assert "one GPU" in str(e.value) and called == []
