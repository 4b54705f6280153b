"""Host logic of the benchmark's end-to-end decode step: the download chunks
and the upload pieces cover every layer once, in order."""

import importlib.util
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_module", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


@pytest.mark.parametrize("L", [1, 2, 3, 4, 5, 17, 24, 32, 64])
def test_download_chunks_cover_the_layers(bench, L):
    sizes = bench.e2e_download_sizes(L)
    assert sum(sizes) == L and all(n >= 1 for n in sizes)
    assert all(n <= 8 for n in sizes)
    # the chunks shrink towards the end; the last one is a single layer
    assert sizes == sorted(sizes, reverse=True) and sizes[-1] == 1


def test_download_chunks_of_32_layers(bench):
    assert bench.e2e_download_sizes(32) == [8, 8, 8, 4, 2, 1, 1]


@pytest.mark.parametrize("L", [1, 2, 3, 4, 5, 32, 64])
def test_upload_pieces_cover_the_layers(bench, L):
    pieces = bench.e2e_upload_pieces(L)
    assert pieces[0] == (0, 1)
    covered = [l for a, b in pieces for l in range(a, b)]
    assert covered == list(range(L))
