"""The top-8 certification's per-lane sort (`route.cu: route_certify_topk`) is a sorting network
of compare-exchange steps `cx(i, j)` (afterwards key[i] >= key[j]).  A comparator network
sorts every input if and only if it sorts every 0-1 input (the 0-1 principle), so checking
the network as written in the source against all 256 0-1 inputs of eight keys, and against
random keys with repeats, proves the descending sort the kernel relies on.  No GPU."""
import itertools
import os
import random
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _network():
    src = open(os.path.join(ROOT, "quantized_grouped_gemm_gb300", "csrc", "route.cu")).read()
    body = src[src.index("auto cx = [&](int i, int j)"):]
    body = body[:body.index("uint32_t top = 0;")]
    net = [(int(a), int(b)) for a, b in re.findall(r"cx\((\d), (\d)\);", body)]
    assert len(net) == 19, net
    return net


def _apply(net, keys):
    k = list(keys)
    for i, j in net:
        hi, lo = max(k[i], k[j]), min(k[i], k[j])
        k[i], k[j] = hi, lo
    return k


def test_network_sorts_every_0_1_input():
    net = _network()
    for bits in itertools.product((0, 1), repeat=8):
        assert _apply(net, bits) == sorted(bits, reverse=True), bits


def test_network_sorts_random_keys_with_repeats():
    net = _network()
    rnd = random.Random(7)
    for _ in range(2000):
        keys = [rnd.randrange(6) for _ in range(8)]
        assert _apply(net, keys) == sorted(keys, reverse=True)


def test_a_broken_network_is_caught():
    # dropping any one comparator leaves some 0-1 input unsorted
    net = _network()
    for drop in range(len(net)):
        broken = net[:drop] + net[drop + 1:]
        assert any(_apply(broken, b) != sorted(b, reverse=True) for b in itertools.product((0, 1), repeat=8)), drop
