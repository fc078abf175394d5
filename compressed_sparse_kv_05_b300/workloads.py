"""The five decode / append workloads this library is measured and checked on.

Shapes only: no arithmetic of the method lives here. Each layer is described by
the same fields the C ABI's ``dsv4_layer_desc`` carries.

  csa_4k        CSA single-layer decode, B=1, 4096-token context, 16 query
                heads over one KV head of 128 dims (64 FP8 + 64 BF16 RoPE),
                separate K and V, ratio 4, indexer 4 heads x 64 dims, top-64,
                window 128. Caches built by streaming the tokens through the
                compressor.
  hca_128k      HCA single-layer decode, B=1, 131072 tokens pooled 128:1 into
                1024 entries, 16 heads, 128 dims, separate K and V, window 128.
  csa_b32_128k  CSA batched decode, B=32, 32768 compressed entries per
                sequence, 64 heads over one shared 512-dim entry (448 FP8 +
                64 BF16), indexer 64 heads x 128 dims, top-512, window 128;
                entries drawn directly, 1% of the blocks carry a planted key.
  compress_1m   one sequence of 2**20 tokens of 512 dims streamed in chunks of
                4096 into a ratio-4 CSA cache (with FP4 indexer keys) and a
                ratio-128 HCA cache.
  stack_1m      eight layers alternating CSA (even) and HCA (odd) at a context
                of 2**20 tokens, B=4, 64 heads, shared 512-dim entry, top-512,
                window 128; each layer's cache drawn from its own seed.
"""
from dataclasses import dataclass, replace
import math


@dataclass(frozen=True)
class Layer:
    kind: str            # "csa" or "hca"
    batch: int
    n_tokens: int        # tokens already in the cache (context length)
    heads: int           # query heads sharing the one KV head
    d_nope: int          # FP8 dims per entry
    d_rope: int          # BF16 RoPE dims per entry
    separate_v: bool     # separate V planes (else V = K)
    ratio: int           # tokens pooled per compressed entry
    window: int          # raw tokens kept in the sliding window
    idx_heads: int = 0   # indexer heads (CSA)
    idx_dim: int = 0     # indexer key dims (CSA)
    topk: int = 0        # compressed entries kept per query (CSA)
    cache_source: str = "stream"   # "stream": built by the compressor; "direct": rows drawn directly
    planted_frac: float = 0.0      # fraction of blocks given a planted indexer key

    @property
    def dim(self):
        return self.d_nope + self.d_rope

    @property
    def n_comp(self):
        return self.n_tokens // self.ratio

    @property
    def sm_scale(self):
        return 1.0 / math.sqrt(self.dim)

    def capacity(self, extra_tokens=0):
        """Compressed-entry capacity that holds the context plus extra_tokens
        appends, rounded up to a multiple of 128 so that every sequence's slice
        of every plane starts on a 16-byte boundary."""
        need = (self.n_tokens + extra_tokens) // self.ratio + 1
        return (need + 127) // 128 * 128


CSA_4K = Layer("csa", 1, 4096, 16, 64, 64, True, 4, 128, idx_heads=4, idx_dim=64, topk=64)
HCA_128K = Layer("hca", 1, 131072, 16, 64, 64, True, 128, 128)
CSA_B32_128K = Layer("csa", 32, 131072, 64, 448, 64, False, 4, 128, idx_heads=64, idx_dim=128,
                     topk=512, cache_source="direct", planted_frac=0.01)
STACK_CSA = Layer("csa", 4, 1 << 20, 64, 448, 64, False, 4, 128, idx_heads=64, idx_dim=128,
                  topk=512, cache_source="direct", planted_frac=0.01)
STACK_HCA = Layer("hca", 4, 1 << 20, 64, 448, 64, False, 128, 128, cache_source="direct")
STACK_1M = tuple(STACK_CSA if l % 2 == 0 else STACK_HCA for l in range(8))

# compress_1m: the same token stream into both caches
COMPRESS_1M_TOKENS = 1 << 20
COMPRESS_1M_CHUNK = 4096
PROJECT_D_MODEL = 4096   # hidden size of the projection workload (the pages give none)
COMPRESS_1M_CSA = Layer("csa", 1, 0, 0, 448, 64, False, 4, 128, idx_dim=128)
COMPRESS_1M_HCA = Layer("hca", 1, 0, 0, 448, 64, False, 128, 128)

WORKLOADS = {
    "csa_4k": (CSA_4K,),
    "hca_128k": (HCA_128K,),
    "csa_b32_128k": (CSA_B32_128K,),
    "stack_1m": STACK_1M,
}


def scaled(layer, **kw):
    """A copy of a layer description with some fields changed (smaller test cases)."""
    return replace(layer, **kw)
