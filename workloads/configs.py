"""The five synthetic workloads: shapes, record formats and selection processes.

Only shapes and generator parameters live here -- nothing of the resolve
method itself.  Both the CPU oracle tests and the GPU path draw their inputs
from the generators in this package, so the two sides always see identical
selections and host records.

Sources on the HiSparse pages:
  * k selected positions per (request, layer, step) out of L_ctx
    ("Inference Systems Infrastructure Notes (6): HiSparse", section 1);
  * B >= k slots per request-layer pair, W_KV x s bytes per record
    (same page, section 2);
  * temporal locality between consecutive steps and cross-layer sharing of
    the anchor's selection (same page, section 4);
  * the uniform-random "falsifier" indexer (Pith review, "What would settle
    it");
  * Quest-style page-granular selection (Pith review, references list).

The numerical knobs (retention fractions, locality window, Zipf exponent,
score drift) are this package's reading of those sources; every value is
stated once, here.
"""
from __future__ import annotations

import dataclasses
from typing import Optional, Tuple

# record value formats
FP16_UNIFORM = 0   # fp16 values ~ U(-1, 1)
BF16_NORMAL = 1    # bf16 values ~ N(0, 1)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    n_requests: int          # R: requests resolved per launch
    n_layers: int            # N_l: sparse layers
    n_positions: int         # L_ctx
    k: int                   # selected positions per (request, layer, step)
    slots: int               # B: GPU hot-cache slots per (request, layer)
    record_bytes: int        # W = W_KV x s
    steps: int               # T: decode steps in the trace
    value_format: int        # FP16_UNIFORM or BF16_NORMAL
    process: str             # "retain", "uniform" or "quest"
    retain: float = 0.0      # fraction of the previous selection kept
    local_frac: float = 0.0  # fraction of new positions drawn near a kept one
    local_window: int = 0    # half-width of the locality window
    # layer -> anchor layer whose selection it shares (None: every layer is
    # its own anchor)
    layer_anchor: Optional[Tuple[int, ...]] = None
    # Quest-style page selection
    page_tokens: int = 0
    always_last_pages: int = 0
    zipf_s: float = 0.0
    score_drift: float = 0.0
    seed: int = 0

    @property
    def anchors(self) -> Tuple[int, ...]:
        if self.layer_anchor is None:
            return tuple(range(self.n_layers))
        return self.layer_anchor

    @property
    def host_bytes(self) -> int:
        return self.n_requests * self.n_layers * self.n_positions * self.record_bytes

    @property
    def cache_bytes(self) -> int:
        return self.n_requests * self.n_layers * self.slots * self.record_bytes

    @property
    def page_table_bytes(self) -> int:
        return self.n_requests * self.n_layers * self.n_positions * 4

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# Tiny CPU-checkable case: 1 request, 1 layer, fp16 W_KV = 64.
TINY = Workload(
    name="tiny", n_requests=1, n_layers=1, n_positions=4096, k=64, slots=128,
    record_bytes=128, steps=100, value_format=FP16_UNIFORM, process="retain",
    retain=0.80, local_frac=0.0, local_window=0)

# DSA / MLA-shaped decode: MLA records of 576 bf16 elements (1152 B).
DSA_MLA = Workload(
    name="dsa_mla", n_requests=8, n_layers=4, n_positions=131072, k=2048,
    slots=4096, record_bytes=1152, steps=256, value_format=BF16_NORMAL,
    process="retain", retain=0.87, local_frac=0.70, local_window=4096)

# Tight cache (B = k) with layers sharing their anchor's selection.
TIGHT_PREFETCH = Workload(
    name="tight_prefetch", n_requests=64, n_layers=8, n_positions=100352,
    k=2048, slots=2048, record_bytes=1152, steps=128,
    value_format=BF16_NORMAL, process="retain", retain=0.85,
    local_frac=0.70, local_window=4096,
    layer_anchor=(0, 0, 0, 0, 4, 4, 4, 4))

# No locality: every step k positions uniform over a 1M-token context.
NO_LOCALITY = Workload(
    name="no_locality", n_requests=8, n_layers=2, n_positions=1 << 20,
    k=2048, slots=4096, record_bytes=1152, steps=64,
    value_format=BF16_NORMAL, process="uniform")

# Quest-style page-granular selection over token records of
# 8 KV heads x 128 dims x (K + V) bf16 = 4096 B.
QUEST_PAGES = Workload(
    name="quest_pages", n_requests=32, n_layers=4, n_positions=32768,
    k=2048, slots=4096, record_bytes=4096, steps=256,
    value_format=BF16_NORMAL, process="quest", page_tokens=16,
    always_last_pages=4, zipf_s=1.1, score_drift=0.05)

ALL = (TINY, DSA_MLA, TIGHT_PREFETCH, NO_LOCALITY, QUEST_PAGES)

# Page-granular records: the Quest selection process over whole pages, each
# page one 64 KiB record (16 tokens x 4096 B), k = 128 pages, B = 256 pages.
QUEST_PAGE_RECORDS = QUEST_PAGES.with_(
    name="quest_page_records", n_positions=2048, k=128, slots=256,
    record_bytes=16 * 4096, page_tokens=1)

BY_NAME = {w.name: w for w in ALL + (QUEST_PAGE_RECORDS,)}
